"""Benchmark of the batched speculative-decoding verify step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c2]
    python bench.py --impl reference ...     # the oracle on the host cores

A step is one verify call over one batch of the workload (all of its rows).
The timed region runs exactly K steps between a barrier and a device
synchronisation, timed with CUDA events on the launching stream; inputs
rotate over enough seeded sets that their total exceeds twice the L2 cache,
so every step reads its logits from HBM. The printed JSON line reports
rows/s (the headline), the achieved HBM bandwidth of the verify kernel
against the measured copy peak, an end-to-end number through the public API
with host buffers, and the oracle timed on the host cores.

With N > 1 (torchrun), each rank runs its own batches on its own GPU (the
sequences of a batch are independent, so the work shards with no
collective); value is the rows of all ranks divided by the slowest rank's
time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, burst copy)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, earlier GB300 measurement)"


# Sources of the kernels the traffic record covers (the verify kernels, the
# LM-head GEMM and the launch decisions made for them); the drafting and
# commit kernels of the decode loop are not in it.
TRAFFIC_SOURCES = ("api.cu", "lmhead.cu", "sv_device.cuh", "sv_launch.h", "verify_common.cuh", "verify_logits.cu",
                   "verify_grouped.cu")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verification_24_gb300", "csrc")
    for name in TRAFFIC_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch from a committed ncu summary, only while the
    kernel sources still hash to the value recorded with the counters."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        entry = d[workload]
        if entry.get("source_hash") != kernel_source_hash():
            return None, "stale (kernel changed since the ncu capture)"
        return float(entry["dram_bytes_per_launch"]), entry.get("note", "")
    except Exception:
        return None, "no ncu capture recorded"


# ----------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background."""

    FIELDS = ("index,timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None
        self.t_marks = []

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def mark(self):
        self.t_marks.append(time.time())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[1].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    rows.append((ts, float(parts[2]), float(parts[3]), parts[5:10]))
                except Exception:
                    continue
        os.unlink(self.file.name)
        if not rows:
            return None
        t0, t1 = (self.t_marks[0], self.t_marks[-1]) if len(self.t_marks) >= 2 else (0, 1e18)
        inside = [r for r in rows if t0 - 1 <= r[0] <= t1 + 1]
        note = "samples within the timed region (1 s timestamp resolution)"
        if not inside:
            inside = rows
            note = "timed region shorter than the sampling interval: samples around it under the same load"
        reasons = set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for r in inside:
            for n, v in zip(names[1:], r[3][1:]):
                if v.strip().lower() in ("active", "1"):
                    reasons.add(n)
        sm = sorted(r[1] for r in inside)
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(r[2] for r in inside),
                "reasons": sorted(reasons), "samples": len(inside), "note": note}


# ----------------------------------------------------------------- workloads


BASE_SEED = {"c1": 0, "c2": 2, "c3": 3, "c4": 4}
RANK_SEED_STRIDE = 1000  # rank r's sets are seeded base + k + 1000 r: its own shard's data


def n_input_sets(name: str, l2_bytes: int) -> tuple:
    """How many seeded input sets a workload rotates over (together more
    than twice the L2, so that every step reads its logits from HBM), and the
    bytes of one set."""
    from synth.workloads import WORKLOADS

    w = WORKLOADS[name]
    esize = 4 if w["dtype"] == "f32" else 2
    B, K, V = w["B"], w["K"], w["V"]
    set_bytes = B * (2 * K + 1) * V * esize
    n_sets = max(2, math.ceil(2 * l2_bytes / set_bytes))
    if name == "c2":  # the sets cycle over the three draft-noise levels
        n_sets = int(math.ceil(n_sets / len(w["tau"])) * len(w["tau"]))
    return n_sets, set_bytes


def make_input_set(name: str, k: int, device, rank: int = 0):
    """Input set k of a workload on `device` (the same generator and seed
    whatever the arm, so both arms read identical logits)."""
    import synth
    from synth.workloads import WORKLOADS

    tau = None
    if name == "c2":
        taus = list(WORKLOADS["c2"]["tau"])
        tau = taus[k % len(taus)]
    return synth.make_workload(name, seed=BASE_SEED[name] + k + RANK_SEED_STRIDE * rank,
                               device=device, tau=tau)


def workload_sets(name: str, device, l2_bytes: int, rank: int = 0):
    """Seeded input sets for a workload, enough that they exceed 2 x L2.
    Each rank gets its own sets (its shard of the global batch)."""
    n_sets, set_bytes = n_input_sets(name, l2_bytes)
    return [make_input_set(name, k, device, rank) for k in range(n_sets)], set_bytes


def acceptance(name: str, n_all: np.ndarray, first: int, count: int, n_sets: int, K: int) -> dict:
    """Mean tokens per verify (accepted drafts + 1) and the fraction of
    sequences that accepted draft i, i = 0..K-1, over the timed steps; for c2
    per draft-noise level tau (the input sets cycle over the three)."""
    from synth.workloads import WORKLOADS

    def stats(rows):
        rows = rows[rows >= 0]
        if rows.size == 0:
            return {}
        return {"sequences": int(rows.size), "mean_tokens_per_verify": float((rows + 1).mean()),
                "accepted_at_position": [float((rows > i).mean()) for i in range(K)]}

    steps = list(range(first, first + count))
    out = {"all": stats(n_all[steps].reshape(-1))}
    if name == "c2":
        taus = list(WORKLOADS["c2"]["tau"])
        for t_i, tau in enumerate(taus):
            sel = [i for i in steps if (i % n_sets) % len(taus) == t_i]
            out[f"tau={tau}"] = stats(n_all[sel].reshape(-1))
    return out


def describe(name: str) -> str:
    return {
        "c1": "B=1 K=4 V=1000 fp32, N(0,3^2)+Zipf(1.1) target, draft=target+N(0,1), T=1",
        "c2": "B=8 K=5 V=32000 fp32 sample T=1, N(0,3^2)+Zipf(1.1) target, "
              "draft=target+N(0,tau^2), tau cycling over {0.3,1.0,3.0}",
        "c3": "B=64 K=4 V=128256 bf16, T=0.8, seqs 0-31 greedy 32-63 sample, "
              "N(0,4^2)+Zipf(1.05) target, draft=0.8*target+N(0,1.5^2)",
        "c4": "B=256 K=8 V=151936 bf16 sample T=1, N(0,4^2)+Zipf(1.1) target, "
              "draft=target+N(0,tau_b^2), tau_b~U[0.2,3.0] per sequence",
    }[name]


def alg_bytes(case, n_accepted: np.ndarray) -> int:
    """Bytes the verify step must read: every target row, the draft rows of
    sample-mode sequences, plus the second pass actually taken (target and
    draft row j after a rejection, target row K for a bonus)."""
    B, K1, V = case.target.shape
    K = K1 - 1
    s = case.target.element_size()
    modes = case.modes.cpu().numpy()
    n_sample = int((modes == 1).sum())
    total = B * K1 * V * s + n_sample * K * V * s
    samp = (modes == 1) & (n_accepted >= 0)
    total += int(((n_accepted < K) & samp).sum()) * 2 * V * s
    total += int(((n_accepted == K) & samp).sum()) * V * s
    return total


def min_bytes(case) -> int:
    B, K1, V = case.target.shape
    s = case.target.element_size()
    n_sample = int((case.modes.cpu().numpy() == 1).sum())
    return B * K1 * V * s + n_sample * (K1 - 1) * V * s


# ----------------------------------------------------------------- ranks


def shard_seq_ids(rank: int, B: int, device) -> torch.Tensor:
    """Global Philox sequence ids of rank `rank`'s shard of B sequences: the
    ranks verify disjoint slices of one global batch, so N ranks draw exactly
    what one GPU would for the whole batch (no collective on the data path)."""
    return torch.arange(rank * B, (rank + 1) * B, dtype=torch.int64, device=device)


def max_over_ranks(x: float, device, world: int) -> float:
    """The largest value over the ranks (the slowest rank's time)."""
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, device, world: int) -> float:
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


def job_rates(rows: float, nbytes: float, ms: float, device, world: int) -> dict:
    """Whole-job rates of one timed region: the rows and algorithmic bytes of
    every rank over the slowest rank's time (each rank's own bytes depend on
    its own accept counts, so they are summed, not multiplied by N)."""
    ms_max = max_over_ranks(ms, device, world)
    rows_all = sum_over_ranks(rows, device, world)
    bytes_all = sum_over_ranks(nbytes, device, world)
    return {"ms_max": ms_max, "rows_per_s": rows_all / (ms_max / 1e3),
            "gbs": bytes_all / (ms_max / 1e3) / 1e9, "rows": rows_all, "bytes": bytes_all}


def bench_config(name: str, B: int, K: int, V: int, n_sets: int, set_bytes: int, l2: int,
                 world: int) -> dict:
    """The workload description both arms print (identical by construction)."""
    return {
        "workload": f"{name}: {describe(name)}",
        "B": B, "K": K, "V": V, "rows_per_step": B * (K + 1),
        "l2": f"inputs rotate over {n_sets} seeded sets "
              f"({n_sets * set_bytes / 2**20:.0f} MiB > 2 x L2 of {l2 / 2**20:.0f} MiB)",
        "parallelism": f"dp x{world}: each rank verifies its own shard of sequences "
                       "(global Philox ids), no collective on the data path",
    }


# ----------------------------------------------------------------- our arm


def uniform_mode(modes: torch.Tensor):
    """'sample' / 'greedy' when every sequence shares the mode (no per-sequence
    array to read), else the per-sequence tensor."""
    m = modes.cpu()
    if bool((m == 1).all()):
        return "sample"
    if bool((m == 0).all()):
        return "greedy"
    return modes


def time_device(sets, steps, warmup, stream, seed0=0, rank=0, overlap=True):
    """Warm-up calls of a workload, and the step function that the timed graph
    captures. Step i verifies input set i % len(sets) with seed seed0 + i and
    writes its own rows of out_tok / out_n (kept for the parity check)."""
    from speculative_decoding_verification_24_gb300 import spec_verify_ex

    B, K1, _ = sets[0].target.shape
    dev = sets[0].target.device
    seq_ids = shard_seq_ids(rank, B, dev)
    out_tok = torch.empty(steps + warmup, B, K1, dtype=torch.int32, device=dev)
    out_n = torch.empty(steps + warmup, B, dtype=torch.int32, device=dev)

    modes = [uniform_mode(c.modes) for c in sets]

    def step(i):
        c = sets[i % len(sets)]
        spec_verify_ex(c.target, c.draft, c.tokens, c.temperature, modes=modes[i % len(sets)],
                       seed=seed0 + i, seq_ids=seq_ids, out_tokens=out_tok[i], out_n_accepted=out_n[i],
                       stream=stream, overlap_previous=overlap)

    with torch.cuda.stream(stream):
        for i in range(warmup):
            step(i)
    torch.cuda.synchronize()
    return step, out_tok, out_n


def capture(step, first, count, stream):
    """A CUDA graph of steps first..first+count-1 (one verify launch each)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(first, first + count):
            step(i)
    torch.cuda.synchronize()
    return g


def replay_ms(graph, stream, label=None):
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    if label:
        torch.cuda.nvtx.range_push(label)
    with torch.cuda.stream(stream):
        start.record(stream)
        graph.replay()
        stop.record(stream)
    torch.cuda.synchronize()
    if label:
        torch.cuda.nvtx.range_pop()
    return start.elapsed_time(stop)


# Timed steps of each sub-result: fixed, whatever --steps the headline runs
# (a sub-result's figure must not move with the headline's step count).
SUB_STEPS = {"c2": 200, "c3": 200, "c4": 100, "c5": 50, "ragged": 100, "tree": 100, "lookup": 200,
             "commit": 200}

HOW_OVERLAPPED = ("independent batches back to back: one CUDA graph of the steps, each launched "
                  "with SV_ARG_OVERLAP_PREVIOUS (programmatic dependent launch: a step streams its "
                  "inputs while the previous step finishes and writes its outputs after that step "
                  "has completed); CUDA events on the launching stream around the replay")
HOW_SERIAL = ("one call at a time, as a decode loop whose next verify depends on this one's "
              "tokens: the same graph of steps launched without SV_ARG_OVERLAP_PREVIOUS, so "
              "each call starts after the previous one has completed")


def launch_plans(sets):
    """The launches of the overlapped and the one-call-at-a-time runs, as the
    library reports them (spec_verify_plan; nothing is enqueued)."""
    from speculative_decoding_verification_24_gb300 import spec_verify_plan

    c = sets[0]
    return {how: spec_verify_plan(c.target, c.draft, c.tokens, c.temperature, modes=uniform_mode(c.modes), seed=0,
                                  overlap_previous=(how == "overlapped"))
            for how in ("overlapped", "serial")}


def logits_timing(sets, steps, warmup, stream, device, world, rank, label):
    """Both timings of a logits workload over the same steps and seeds:
    overlapped (independent batches back to back) and serial (one call at a
    time). Returns the two times, the outputs of the overlapped run and
    whether the serial run emitted the same tokens (it must: same inputs,
    same seeds)."""
    step, out_tok, out_n = time_device(sets, steps, warmup, stream, rank=rank)
    graph = capture(step, warmup, steps, stream)
    replay_ms(graph, stream)  # warm replay: same launches, same inputs
    res = {"step": step, "graph": graph, "out_tok": out_tok, "out_n": out_n}
    res["ms"] = replay_ms(graph, stream, f"{label} overlapped x{steps}")
    s_step, s_tok, s_n = time_device(sets, steps, warmup, stream, rank=rank, overlap=False)
    s_graph = capture(s_step, warmup, steps, stream)
    replay_ms(s_graph, stream)
    res["serial_ms"] = replay_ms(s_graph, stream, f"{label} serial x{steps}")
    del s_graph
    sl = slice(warmup, warmup + steps)
    same = (out_tok[sl] == s_tok[sl]).all(dim=2) & (out_n[sl] == s_n[sl])
    # the two runs may use different cluster sizes, so their float32 sums
    # differ in rounding and may decide a near-tie differently; the oracle
    # leg checks both runs
    res["serial_differing"] = int((~same).sum())
    res["serial_tok"], res["serial_n"] = s_tok, s_n
    return res


def run_ours(args, rank, world, device):
    from speculative_decoding_verification_24_gb300.build import build

    build()
    props = torch.cuda.get_device_properties(device)
    l2 = int(getattr(props, "L2_cache_size", 0) or 129 * 2**20)
    sets, set_bytes = workload_sets(args.workload, device, l2, rank)
    case0 = sets[0]
    B, K1, V = case0.target.shape
    rows_per_step = B * K1
    stream = torch.cuda.Stream(device)
    t = logits_timing(sets, args.steps, args.warmup, stream, device, world, rank, args.workload)
    plans = launch_plans(sets)
    graph = t["graph"]

    sampler = ClockSampler(device.index if device.index is not None else 0)
    sampler.start()
    # keep the GPU busy briefly so the sampler sees clocks under this load
    t_end = time.time() + 0.5
    while time.time() < t_end:
        replay_ms(graph, stream)

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.mark()
    ms = replay_ms(graph, stream, f"timed: {args.workload} x{args.steps}")
    sampler.mark()
    if world > 1:
        torch.distributed.barrier()
    time.sleep(0.25)
    clocks = sampler.stop()
    del graph, t["graph"]

    # eager launches from Python, for comparison (not the headline)
    e_start = torch.cuda.Event(enable_timing=True)
    e_stop = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e_start.record(stream)
    with torch.cuda.stream(stream):
        for i in range(args.warmup, args.warmup + args.steps):
            t["step"](i)
    e_stop.record(stream)
    torch.cuda.synchronize()
    eager_ms = max_over_ranks(e_start.elapsed_time(e_stop), device, world)

    # exact algorithmic bytes of every timed step, from its own outputs
    n_all = t["out_n"].cpu().numpy()
    timed = range(args.warmup, args.warmup + args.steps)
    bytes_alg = sum(alg_bytes(sets[i % len(sets)], n_all[i]) for i in timed)
    bytes_min = sum(min_bytes(sets[i % len(sets)]) for i in timed)
    job = job_rates(rows_per_step * args.steps, bytes_alg, ms, device, world)
    serial = job_rates(rows_per_step * args.steps, bytes_alg, t["serial_ms"], device, world)
    ms_max = job["ms_max"]
    gbs = job["gbs"]
    peak, peak_src = measured_peaks()
    traffic, traffic_note = profiled_traffic(args.workload)
    cfg = bench_config(args.workload, B, K1 - 1, V, len(sets), set_bytes, l2, world)

    result = {
        "metric": "verify rows/s",
        "value": job["rows_per_s"],
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_max / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "input_dtype": "f32" if case0.target.dtype == torch.float32 else "bf16",
        "data": "synthetic (seeded generators in synth/; no dataset or weights)",
        "config": cfg,
        "hbm_gbs": gbs,
        "hbm_bytes_per_step": job["bytes"] / args.steps / world,
        "roofline": {
            "bound": "hbm",
            "kernel": "sv::verify_logits_kernel",
            "achieved": gbs / world,
            "peak": peak,
            "unit": "GB/s",
            "frac": gbs / world / peak,
            "peak_source": peak_src,
            "frac_of_nominal_8tbs": gbs / world / NOMINAL_HBM_GBS,
            "traffic": None if traffic is None else traffic,
            "traffic_note": traffic_note,
            "algorithmic_bytes_per_launch": bytes_alg / args.steps,
            "min_bytes_per_launch": bytes_min / args.steps,
            "timing": "CUDA events on the launching stream over the timed region / steps",
        },
        "gpu_launches": args.steps,
        "clocks": clocks,
        "timing": "value: " + HOW_OVERLAPPED,
        "serial": {"ms_per_step": serial["ms_max"] / args.steps,
                   "rows_per_s": serial["rows_per_s"],
                   "hbm_gbs": serial["gbs"],
                   "frac_of_measured_peak": serial["gbs"] / world / peak,
                   "frac_of_nominal_8tbs": serial["gbs"] / world / NOMINAL_HBM_GBS,
                   "sequences_differing_from_overlapped": t["serial_differing"],
                   "plan": plans["serial"],
                   "how": HOW_SERIAL},
        "plan": plans["overlapped"],
        "eager_rows_per_s": world * rows_per_step * args.steps / (eager_ms / 1e3),
    }
    result["acceptance"] = acceptance(args.workload, n_all, args.warmup, args.steps, len(sets), K1 - 1)
    result["e2e"] = run_e2e(args, sets, device, stream, world, rank)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        base, check = oracle_leg(sets, t["out_tok"], t["out_n"], args.warmup, args.steps,
                                 args.cpu_seconds, rank, serial=(t["serial_tok"], t["serial_n"]))
        result["cpu_baseline"] = base
        result["parity"] = check
    if rank == 0 and not args.no_extra and world == 1:
        result["other_workloads"] = other_workloads(args, device, l2, stream)
    return result


def run_e2e(args, sets, device, stream, world, rank=0):
    """Same metric through the public API with host buffers. Every step copies
    its inputs from pinned host memory into one of two device buffers (on a
    copy stream, so that step i+1's copy overlaps step i's verify), verifies
    them with spec_verify_ex and copies the results back to pinned host
    memory. The K steps run from one CUDA graph, as a serving loop would
    replay them; the plain eager loop on one stream is reported beside it."""
    from speculative_decoding_verification_24_gb300 import spec_verify_ex

    n_host = min(len(sets), 4)
    seq_ids = shard_seq_ids(rank, sets[0].target.shape[0], device)
    host = []
    for c in sets[:n_host]:
        host.append(tuple(t.cpu().pin_memory() for t in (c.target, c.draft, c.tokens, c.modes)))
    c0 = sets[0]
    B, K1, _ = c0.target.shape
    bufs = [tuple(torch.empty_like(t) for t in (c0.target, c0.draft, c0.tokens, c0.modes))
            for _ in range(2)]
    outs = [(torch.empty(B, K1, dtype=torch.int32, device=device),
             torch.empty(B, dtype=torch.int32, device=device)) for _ in range(2)]
    res = [(torch.empty(B, K1, dtype=torch.int32).pin_memory(),
            torch.empty(B, dtype=torch.int32).pin_memory()) for _ in range(2)]
    mode0 = uniform_mode(c0.modes)
    h2d = sum(t.numel() * t.element_size() for t in host[0])
    d2h = res[0][0].numel() * 4 + res[0][1].numel() * 4
    copy_stream = torch.cuda.Stream(device)

    def verify(i, k, on):
        dt, dd, dx, dm = bufs[k]
        spec_verify_ex(dt, dd, dx, c0.temperature, modes=dm if isinstance(mode0, torch.Tensor) else mode0,
                       seed=i, seq_ids=seq_ids, out_tokens=outs[k][0], out_n_accepted=outs[k][1], stream=on)
        res[k][0].copy_(outs[k][0], non_blocking=True)
        res[k][1].copy_(outs[k][1], non_blocking=True)

    def load(i, k):
        for dst, src in zip(bufs[k], host[i % n_host]):
            dst.copy_(src, non_blocking=True)

    # eager, one stream: copy, verify, read back, step after step
    def eager_step(i):
        load(i, 0)
        verify(i, 0, stream)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            eager_step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            eager_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    eager_ms = max_over_ranks(e0.elapsed_time(e1), device, world)

    # pipelined graph of K steps: copies on copy_stream, verifies on stream
    def pipelined(first, n):
        copied = [torch.cuda.Event() for _ in range(n)]
        done = [torch.cuda.Event() for _ in range(n)]
        copy_stream.wait_stream(stream)
        for t in range(n):
            i, k = first + t, t % 2
            with torch.cuda.stream(copy_stream):
                if t >= 2:
                    copy_stream.wait_event(done[t - 2])  # buffer k is free again
                load(i, k)
                copied[t].record(copy_stream)
            stream.wait_event(copied[t])
            verify(i, k, stream)
            done[t].record(stream)
        stream.wait_stream(copy_stream)

    with torch.cuda.stream(stream):
        pipelined(0, max(2, args.warmup))
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        pipelined(args.warmup, args.steps)
    torch.cuda.synchronize()
    ms = replay_ms(g, stream)  # the first replay loads the graph
    ms = max_over_ranks(replay_ms(g, stream, "timed: e2e"), device, world)
    rows = world * B * K1 * args.steps
    pipelined = {"value": rows / (ms / 1e3), "ms_per_step": ms / args.steps,
                 "how": "the K steps replayed from one CUDA graph: each step's inputs copied "
                        "from pinned host memory into one of two device buffers on a copy "
                        "stream (step i+1's copy overlaps step i's verify), spec_verify_ex, "
                        "its results copied back to pinned host memory"}
    eager = {"value": rows / (eager_ms / 1e3), "ms_per_step": eager_ms / args.steps,
             "how": "the K steps launched eagerly on one stream: copy in, spec_verify_ex, "
                    "copy out, step after step"}
    best = "pipelined_graph" if pipelined["value"] >= eager["value"] else "eager_one_stream"
    best_ms = ms if best == "pipelined_graph" else eager_ms
    return {"value": max(pipelined["value"], eager["value"]), "unit": "rows/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "h2d_gbs": h2d * args.steps / (best_ms / 1e3) / 1e9,
            "method": best, "pipelined_graph": pipelined, "eager_one_stream": eager,
            "how": "every step copies its inputs from pinned host memory and its results "
                   "back, through the public API (spec_verify_ex); CUDA events around the K "
                   "steps; value is the faster of the two methods below"}


def oracle_leg(sets, out_tok, out_n, first, count, seconds, rank=0, target_of=None, serial=None):
    """The cpu_baseline leg: the oracle as it stands, timed on the host cores
    (threads over sequences) on the timed steps of the GPU run, in order and
    with the same seeds and sequence ids, until about `seconds` of oracle
    time; then its outputs for those steps compared with the GPU's.

    Returns (cpu_baseline, parity). parity counts the sequences checked, the
    exact matches and the near-ties, split into accept-test ties and draw
    ties (bands in oracle/parity.py), and must show no mismatch outside them.
    target_of(i) optionally gives step i's target rows (the LM-head path
    verifies the GPU's own fp32 logits)."""
    from oracle import oracle as orc
    from oracle import parity as par
    from synth.workloads import to_numpy_logits

    cores = os.cpu_count() or 1
    host = {}
    tok_all = out_tok.cpu().numpy()
    n_all = out_n.cpu().numpy()
    ser = None if serial is None else (serial[0].cpu().numpy(), serial[1].cpu().numpy())
    ser_tot = {"sequences": 0, "near_tie_mismatches": 0, "mismatches": 0}
    rows = calls = used = 0
    el = 0.0
    tot = {"steps_checked": 0, "sequences": 0, "exact": 0, "accept_near_ties": 0, "draw_near_ties": 0,
           "near_tie_mismatches": 0, "mismatches": 0}
    first_bad = []
    for t in range(count):
        if el >= seconds:
            break
        i = first + t
        k = i % len(sets)
        c = sets[k]
        if k not in host:
            host[k] = (to_numpy_logits(c.draft), c.tokens.cpu().numpy(), c.modes.cpu().numpy())
        drf, tok, modes = host[k]
        tgt = to_numpy_logits(c.target) if target_of is None else target_of(i)
        B, K1, _ = tgt.shape
        threads = min(cores, B)
        used = max(used, threads)
        ids = shard_seq_ids(rank, B, "cpu").numpy().astype(np.uint64)
        t1 = time.perf_counter()
        ref = orc.verify(tgt, drf, tok, c.temperature, modes, seed=i, seq_ids=ids, threads=threads)
        el += time.perf_counter() - t1
        rows += B * K1
        calls += 1
        acc_tie = ref["accept_margin"] < par.ACCEPT_TIE_REL
        draw_tie = ~acc_tie & par.near_ties(ref)
        cmp = par.compare(tok_all[i], n_all[i], ref, ties=acc_tie | draw_tie)
        tot["steps_checked"] += 1
        tot["sequences"] += cmp["sequences"]
        tot["accept_near_ties"] += int(acc_tie.sum())
        tot["draw_near_ties"] += int(draw_tie.sum())
        tot["near_tie_mismatches"] += cmp["near_tie_mismatches"]
        tot["mismatches"] += cmp["mismatches"]
        tot["exact"] += cmp["sequences"] - cmp["near_tie_mismatches"] - cmp["mismatches"]
        if ser is not None:
            sc = par.compare(ser[0][i], ser[1][i], ref, ties=acc_tie | draw_tie)
            for key in ser_tot:
                ser_tot[key] += sc[key]
        first_bad += [dict(step=i, **m) for m in cmp["first_mismatches"]][:3 - len(first_bad)]
    base = {"value": rows / el if el > 0 else None, "unit": "rows/s", "cores": used, "kind": "oracle",
            "sample": f"the first {calls} timed steps ({rows} rows), same inputs, seeds and sequence "
                      f"ids as the GPU run; {el:.1f} s of oracle time, threads over sequences"}
    tot["near_tie_fraction"] = (tot["accept_near_ties"] + tot["draw_near_ties"]) / max(1, tot["sequences"])
    tot["bands"] = {"accept": f"|u*P_d(x) - P_t(x)| < {par.ACCEPT_TIE_REL:g} * P_d(x)",
                    "draw": f"t within {par.DRAW_TIE_ABS:g} of an edge of the chosen token's "
                            "cumulative interval (probability units)"}
    tot["how"] = ("the oracle (double precision, own Philox) on the GPU's timed steps; tokens and "
                  "accept counts compared exactly outside the near-tie bands")
    if ser is not None:
        tot["serial_run"] = dict(ser_tot, how="the one-call-at-a-time run's outputs for the same steps, "
                                               "against the same oracle outputs")
    if first_bad:
        tot["first_mismatches"] = first_bad
    return base, tot


SUB_ORACLE_SECONDS = 3.0  # oracle time per sub-result's parity check


def other_workloads(args, device, l2, stream):
    """The other workloads, each measured the same way over its own fixed
    number of steps (SUB_STEPS), with the oracle's check of its outputs."""
    out = {}
    for name in args.also:
        if name == args.workload:
            continue
        if name == "c5":
            try:
                out[name] = lmhead_workload(args, device, stream)
            except Exception as e:  # report, do not hide
                out[name] = {"error": repr(e)}
            torch.cuda.empty_cache()
            continue
        if name in NEXT_ROW_NAMES:
            try:
                out[name] = next_row_workload(name, args, device, l2, stream)
            except Exception as e:  # report, do not hide
                out[name] = {"error": repr(e)}
            torch.cuda.empty_cache()
            continue
        try:
            sets, set_bytes = workload_sets(name, device, l2)
            steps = SUB_STEPS[name]
            t = logits_timing(sets, steps, args.warmup, stream, device, 1, 0, name)
            del t["graph"]
            ms, serial_ms = t["ms"], t["serial_ms"]
            n_all = t["out_n"].cpu().numpy()
            ba = sum(alg_bytes(sets[i % len(sets)], n_all[i])
                     for i in range(args.warmup, args.warmup + steps))
            B, K1, V = sets[0].target.shape
            gbs = ba / (ms / 1e3) / 1e9
            peak, _ = measured_peaks()
            traffic, traffic_note = profiled_traffic(name)
            out[name] = {"workload": describe(name), "steps": steps,
                         "traffic": traffic, "traffic_note": traffic_note,
                         "algorithmic_bytes_per_launch": ba / steps,
                         "rows_per_s": B * K1 * steps / (ms / 1e3), "us_per_step": ms * 1e3 / steps,
                         "hbm_gbs": gbs, "frac_of_measured_peak": gbs / peak,
                         "frac_of_nominal_8tbs": gbs / NOMINAL_HBM_GBS,
                         "how": HOW_OVERLAPPED,
                         "serial": {"us_per_step": serial_ms * 1e3 / steps,
                                    "rows_per_s": B * K1 * steps / (serial_ms / 1e3),
                                    "frac_of_measured_peak": ba / (serial_ms / 1e3) / 1e9 / peak,
                                    "frac_of_nominal_8tbs": ba / (serial_ms / 1e3) / 1e9 / NOMINAL_HBM_GBS,
                                    "sequences_differing_from_overlapped": t["serial_differing"],
                                    "plan": launch_plans(sets)["serial"],
                                    "how": HOW_SERIAL},
                         "plan": launch_plans(sets)["overlapped"],
                         "acceptance": acceptance(name, n_all, args.warmup, steps, len(sets), K1 - 1),
                         "input_sets": len(sets)}
            if not args.no_cpu_baseline:
                out[name]["cpu_baseline"], out[name]["parity"] = oracle_leg(
                    sets, t["out_tok"], t["out_n"], args.warmup, steps, SUB_ORACLE_SECONDS,
                    serial=(t["serial_tok"], t["serial_n"]))
            del sets, t
            torch.cuda.empty_cache()
        except Exception as e:  # report, do not hide
            out[name] = {"error": repr(e)}
    return out


NEXT_ROW_NAMES = ("ragged", "tree", "lookup", "commit")


def timed_graph_ms(step, args, steps, stream):
    """Warm-up calls, then one CUDA graph of `steps` calls replayed twice; the
    second replay's time (CUDA events on the launching stream)."""
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    torch.cuda.synchronize()
    graph = capture(step, args.warmup, steps, stream)
    replay_ms(graph, stream)
    ms = replay_ms(graph, stream)
    del graph
    return ms


def next_row_workload(name, args, device, l2, stream):
    """The decode-loop pieces around the verify step, each on its own seeded
    inputs (sizes in synth.NEXT_ROWS): ragged draft counts on c4's shapes,
    greedy tree verification, prompt lookup and the commit step."""
    import synth
    from speculative_decoding_verification_24_gb300 import (spec_commit, spec_prompt_lookup,
                                                            spec_verify_ex, spec_verify_tree)

    cfg = synth.NEXT_ROWS[name]
    steps = SUB_STEPS[name]
    peak, _ = measured_peaks()

    def hbm(nbytes, ms):
        gbs = nbytes / (ms / 1e3) / 1e9
        return {"hbm_gbs": gbs, "frac_of_measured_peak": gbs / peak, "frac_of_nominal_8tbs": gbs / NOMINAL_HBM_GBS}

    if name == "ragged":
        sets, _ = workload_sets(cfg["base"], device, l2)
        B, K1, V = sets[0].target.shape
        K = K1 - 1
        s = sets[0].target.element_size()
        lens = [synth.make_draft_lens(B, K, seed=400 + k, device=device) for k in range(len(sets))]
        out_t = torch.empty(args.warmup + steps, B, K1, dtype=torch.int32, device=device)
        out_n = torch.empty(args.warmup + steps, B, dtype=torch.int32, device=device)

        def step(i):
            c = sets[i % len(sets)]
            spec_verify_ex(c.target, c.draft, c.tokens, c.temperature, modes="sample", seed=i,
                           out_tokens=out_t[i], out_n_accepted=out_n[i], stream=stream,
                           overlap_previous=True, draft_lens=lens[i % len(sets)])

        ms = timed_graph_ms(step, args, steps, stream)
        n_all = out_n.cpu().numpy()
        nbytes, rows = 0, 0
        for i in range(args.warmup, args.warmup + steps):
            kb = lens[i % len(sets)].cpu().numpy().astype(np.int64)
            n = n_all[i]
            rows += int((kb + 1).sum())
            nbytes += int(((2 * kb + 1) * V * s).sum())            # rows 0..Kb of both
            nbytes += int(((n >= 0) & (n < kb)).sum()) * 2 * V * s  # residual row pair
            nbytes += int((n == kb).sum()) * V * s                  # bonus row
        del sets
        return {"workload": "c4's shapes (B=256, K=8, V=151936 bf16, sample) with per-sequence "
                            "draft counts uniform over 0..8", "steps": steps,
                "rows_per_s": rows / (ms / 1e3), "us_per_step": ms * 1e3 / steps,
                "algorithmic_bytes_per_launch": nbytes / steps, **hbm(nbytes / steps, ms / steps),
                "how": "overlapped calls (SV_ARG_OVERLAP_PREVIOUS) from one CUDA graph, inputs rotating over > 2 x L2"}

    if name == "tree":
        B, N, V = cfg["B"], cfg["N"], cfg["V"]
        one = B * N * V * 2
        n_sets = max(2, math.ceil(2 * l2 / one))
        sets = [synth.make_tree_case(B, N, V, cfg["dtype"], cfg["sigma_t"], cfg["zipf_s"], cfg["p_follow"],
                                     seed=600 + k, device=device) for k in range(n_sets)]
        outs = (torch.empty(B, N, dtype=torch.int32, device=device), torch.empty(B, dtype=torch.int32, device=device),
                torch.empty(B, dtype=torch.int32, device=device))

        def step(i):
            t, x, par = sets[i % n_sets]
            spec_verify_tree(t, x, par, out_tokens=outs[0], out_n_accepted=outs[1], out_last_node=outs[2],
                             stream=stream)

        ms = timed_graph_ms(step, args, steps, stream)
        mean_acc = float(outs[1].float().mean())
        del sets
        return {"workload": f"greedy tree verify: {B} trees of {N} nodes, V={V} bf16 rows "
                            "(N(0,4^2)+Zipf(1.05); a node takes its parent's top token with p=0.6)",
                "steps": steps, "rows_per_s": B * N * steps / (ms / 1e3), "us_per_step": ms * 1e3 / steps,
                "algorithmic_bytes_per_launch": one, **hbm(one, ms / steps),
                "mean_accepted_depth_last_step": mean_acc,
                "how": "plain calls from one CUDA graph (every row read once), inputs rotating over > 2 x L2"}

    if name == "lookup":
        B, L, vocab = cfg["B"], cfg["L_max"], cfg["vocab"]
        tok0, lens0 = synth.make_contexts(B, L, vocab, seed=700, copy_prob=cfg["copy_prob"])
        n_sets = max(2, math.ceil(2 * l2 / (B * L * 4)))
        # further sets: the same structure with token ids shifted and rows rolled
        sets = [(torch.from_numpy(np.roll((tok0 + 7 * k) % vocab, k, axis=0)).to(device),
                 torch.from_numpy(np.roll(lens0, k)).to(device)) for k in range(n_sets)]
        out_d = torch.empty(B, cfg["n_drafts"], dtype=torch.int32, device=device)
        out_n = torch.empty(B, dtype=torch.int32, device=device)

        def step(i):
            ctx, ln = sets[i % n_sets]
            spec_prompt_lookup(ctx, ln, cfg["max_ngram"], cfg["n_drafts"], out_drafts=out_d, out_n_drafts=out_n,
                               stream=stream)

        ms = timed_graph_ms(step, args, steps, stream)
        nbytes = sum(int(sets[i % n_sets][1].clamp(min=0).sum()) * 4
                     for i in range(args.warmup, args.warmup + steps)) / steps
        found = int((out_n > 0).sum())
        del sets
        return {"workload": f"prompt lookup: {B} contexts of up to {L} tokens (vocab {vocab}, "
                            f"lengths uniform), n-grams up to {cfg['max_ngram']}, {cfg['n_drafts']} drafts",
                "steps": steps, "contexts_per_s": B * steps / (ms / 1e3), "us_per_step": ms * 1e3 / steps,
                "algorithmic_bytes_per_launch": nbytes, **hbm(nbytes, ms / steps),
                "sequences_with_drafts_last_step": found,
                "how": "plain calls from one CUDA graph; each context's tokens read once is the "
                       "algorithmic traffic; inputs rotating over > 2 x L2"}

    if name == "commit":
        B, L, K = cfg["B"], cfg["L_max"], cfg["K"]
        rng = np.random.default_rng(800)
        ctx = torch.zeros(B, L, dtype=torch.int32, device=device)
        start = torch.full((B,), L // 2, dtype=torch.int32, device=device)
        lens = start.clone()
        n_var = 8
        toks = [torch.from_numpy(rng.integers(0, 32000, (B, K + 1)).astype(np.int32)).to(device) for _ in range(n_var)]
        nacc = [torch.from_numpy(rng.integers(0, K + 1, B).astype(np.int32)).to(device) for _ in range(n_var)]
        out_c = torch.empty(B, dtype=torch.int32, device=device)

        def step(i):
            spec_commit(ctx, lens, toks[i % n_var], nacc[i % n_var], out_n_committed=out_c, stream=stream)

        with torch.cuda.stream(stream):
            for i in range(args.warmup):
                step(i)
        torch.cuda.synchronize()
        graph = capture(step, args.warmup, steps, stream)
        lens.copy_(start)
        replay_ms(graph, stream)
        lens.copy_(start)
        ms = replay_ms(graph, stream)
        del graph
        moved = B * (K + 1) * 4 * 2 + B * 4 * 3
        return {"workload": f"commit: {B} contexts of {L} slots, K={K} (up to {K + 1} tokens appended "
                            "per sequence)", "steps": steps, "us_per_step": ms * 1e3 / steps,
                "calls_per_s": steps / (ms / 1e3), "bytes_per_launch": moved,
                "bound": "launch latency (a few KB per call)",
                "how": "plain calls from one CUDA graph"}
    raise ValueError(name)


def lmhead_workload(args, device, stream, n_sets=4):
    """The fused LM-head workload (hidden [32, 6, 4096] bf16, W [4096, 128256]
    bf16): spec_verify_lmhead per step, and the tensor-core GEMM alone. W
    (1.05 GB) is far larger than L2, so every step streams it from HBM."""
    import synth
    from speculative_decoding_verification_24_gb300 import (spec_lmhead_logits, spec_verify_lmhead,
                                                            spec_verify_lmhead_workspace_bytes)
    from synth.workloads import WORKLOADS

    w = WORKLOADS["c5"]
    base = synth.make_workload("c5", seed=5, device=device)
    sets = [base] + [synth.make_lmhead_case(B=w["B"], K=w["K"], V=w["V"], d=w["d"], seed=5 + k,
                                            device=device) for k in range(1, n_sets)]
    W = base.W  # one head, as in serving: the hidden states and drafts change per step
    B, K1, d = base.hidden.shape
    K, V = K1 - 1, W.shape[1]
    M = B * K1
    steps = SUB_STEPS["c5"]
    ws = torch.empty(spec_verify_lmhead_workspace_bytes(B, K, d, V), dtype=torch.uint8, device=device)
    out_t = torch.empty(steps + args.warmup, B, K1, dtype=torch.int32, device=device)
    out_n = torch.empty(steps + args.warmup, B, dtype=torch.int32, device=device)
    logits = torch.empty(M, V, dtype=torch.float32, device=device)
    hid2d = [c.hidden.reshape(M, d) for c in sets]

    def fused(i):
        c = sets[i % n_sets]
        spec_verify_lmhead(c.hidden, W, c.draft, c.tokens, c.temperature, seed=i, workspace=ws,
                           out_tokens=out_t[i], out_n_accepted=out_n[i], stream=stream)

    def gemm(i):
        spec_lmhead_logits(hid2d[i % n_sets], W, out=logits, stream=stream)

    res = {"workload": "c5: fused LM head + verify, hidden [B=32, K+1=6, d=4096] bf16 ~ N(0,1), "
                       "W [4096, 128256] bf16 ~ N(0, 0.02^2), draft = hidden.W + N(0,1) (bf16), "
                       "T=1, sample mode",
           "steps": steps, "l2": f"W of {d * V * 2 / 2**30:.2f} GiB streams from HBM every step; "
                                 f"hidden and draft rotate over {n_sets} sets"}
    timings = {}
    for name, fn in (("fused", fused), ("gemm", gemm)):
        with torch.cuda.stream(stream):
            for i in range(args.warmup):
                fn(i)
        torch.cuda.synchronize()
        g = capture(fn, args.warmup, steps, stream)
        replay_ms(g, stream)
        timings[name] = replay_ms(g, stream) / steps
        del g
    peak, peak_src = measured_peaks()
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tf_peak = float(json.load(f)["bf16_tflops"])
        tf_src = "measured (MEASURED_PEAKS.json bf16_tflops, burst cuBLAS)"
    except Exception:
        tf_peak, tf_src = 1900.0, "fallback (1.9 PFLOP/s bf16 burst, earlier GB300 measurement)"
    g_ms, f_ms = timings["gemm"], timings["fused"]
    w_bytes = d * V * 2
    io_bytes = w_bytes + M * d * 2 + M * V * 4
    flops = 2.0 * M * d * V
    n_all = out_n[args.warmup:args.warmup + steps].cpu().numpy()
    res.update({
        "rows_per_s": M / (f_ms / 1e3), "us_per_step": f_ms * 1e3,
        "gemm_us": g_ms * 1e3, "verify_us": (f_ms - g_ms) * 1e3,
        "verify_us_means": "the fused step minus the GEMM alone (spec_lmhead_logits): the epilogue's "
                           "tile partials, the draft rows' partials and the verify launch after the GEMM",
        "fused_step_w_stream": {
            "achieved": w_bytes / (f_ms / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
            "frac": w_bytes / (f_ms / 1e3) / 1e9 / peak, "peak_source": peak_src,
            "what": "the whole fused step (GEMM with epilogue partials, then the verify) against the "
                    "W-streaming roofline (d*V*2 bytes per step)"},
        "mean_tokens_per_verify": float((n_all + 1).mean()),
        "roofline": {
            "bound": "hbm", "kernel": "sv::lmhead_gemm_kernel",
            "achieved": w_bytes / (g_ms / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
            "frac": w_bytes / (g_ms / 1e3) / 1e9 / peak, "peak_source": peak_src,
            "algorithmic_bytes_per_launch": w_bytes,
            "what": "W-streaming roofline: the head's weights (d*V*2 bytes) once per launch",
            "all_io_gbs": io_bytes / (g_ms / 1e3) / 1e9,
        },
        "tensor": {"achieved_tflops": flops / (g_ms / 1e3) / 1e12, "peak_tflops": tf_peak,
                   "frac": flops / (g_ms / 1e3) / 1e12 / tf_peak, "peak_source": tf_src,
                   "note": "M = B*(K+1) = 192 rows make the product HBM-bound by design"},
        "gpu_launches_per_step": 2,
    })
    if not args.no_cpu_baseline:
        # the last timed step, checked against the oracle run on the GPU's
        # own fp32 logits (still in the workspace) and the same draft rows
        last = args.warmup + steps - 1
        gpu_logits = ws[:M * V * 4].view(torch.float32).reshape(B, K1, V)
        res["cpu_baseline"], res["parity"] = oracle_leg(
            sets, out_t, out_n, last, 1, SUB_ORACLE_SECONDS, target_of=lambda i: gpu_logits.cpu().numpy())
        res["parity"]["how"] = ("the oracle on the last timed step's fp32 logits as the GEMM wrote "
                                "them (the workspace) and the same bf16 draft rows; tokens and accept "
                                "counts compared exactly outside the near-tie bands")
    del sets, ws, logits
    torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------------- reference arm


def run_reference(args):
    """The reference arm: the oracle, as it stands, timed on the host cores on
    this workload. It reads the same input sets as the GPU arm (same
    generator, seeds and device), cycles over them step by step with the same
    seeds, and verifies a bounded sample of each batch (its first n_seq
    sequences) so that the whole run stays within a few minutes."""
    from oracle import oracle as orc
    from synth.workloads import to_numpy_logits

    orc.build()
    gen_dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    l2 = 129 * 2**20
    if gen_dev.type == "cuda":
        l2 = int(getattr(torch.cuda.get_device_properties(gen_dev), "L2_cache_size", 0) or l2)
    n_sets, set_bytes = n_input_sets(args.workload, l2)
    host = []
    for k in range(n_sets):
        c = make_input_set(args.workload, k, gen_dev)
        host.append((to_numpy_logits(c.target), to_numpy_logits(c.draft), c.tokens.cpu().numpy(),
                     c.modes.cpu().numpy(), c.temperature))
        del c
    if gen_dev.type == "cuda":
        torch.cuda.empty_cache()
    B, K1, V = host[0][0].shape
    cores = os.cpu_count() or 1
    threads = min(cores, B)
    ids = np.arange(B, dtype=np.uint64)

    def call(i, n_seq):
        tgt, drf, tok, modes, T = host[i % n_sets]
        orc.verify(tgt, drf, tok, T, modes, seed=i, seq_ids=ids, threads=min(threads, n_seq),
                   seq_range=(0, n_seq))

    # size the per-step sample from one timed call of a few sequences
    budget_s = 1.0
    probe = min(B, threads)
    t0 = time.perf_counter()
    call(0, probe)
    per_seq = (time.perf_counter() - t0) / probe * min(threads, B)
    n_seq = B if per_seq * B / threads <= budget_s else max(1, int(budget_s * threads / per_seq))
    n_seq = min(B, max(n_seq, 1))
    for i in range(args.warmup):
        call(i, n_seq)
    t0 = time.perf_counter()
    for i in range(args.warmup, args.warmup + args.steps):
        call(i, n_seq)
    el = time.perf_counter() - t0
    value = n_seq * K1 * args.steps / el
    sample = (f"the first {n_seq} of {B} sequences of each step's batch ({n_seq * K1} rows), "
              f"{args.steps} steps over the same input sets and seeds as the GPU arm")
    return {
        "impl": "reference", "metric": "verify rows/s", "value": value, "unit": "rows/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded generators in synth/; no dataset or weights)",
        "config": bench_config(args.workload, B, K1 - 1, V, n_sets, set_bytes, l2, args.gpus),
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": min(threads, n_seq),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "note": "the reference arm is the plain C double-precision oracle (the pages print no "
                "implementation of the verify step to install); under torchrun rank 0 alone runs it",
    }


def profile_run(args, device):
    """--profile NAME: warmup + steps eager calls of one workload and no bench
    line, for ncu (every launch of the verify kernel, launched as the bench
    times it, with SV_ARG_OVERLAP_PREVIOUS and so the same cluster size; or
    for c5 the LM-head GEMM then the verify kernel; inputs larger than L2).
    NAME-alone: the same calls without the flag, as the bench's one-call-at-a-
    time block launches them (c3: the grouped kernel)."""
    from speculative_decoding_verification_24_gb300 import (spec_verify_ex, spec_verify_lmhead,
                                                            spec_verify_lmhead_workspace_bytes)
    from speculative_decoding_verification_24_gb300.build import build

    build()
    n = args.warmup + args.steps
    if args.profile == "c5":
        import synth
        c = synth.make_workload("c5", seed=5, device=device)
        B, K1, d = c.hidden.shape
        ws = torch.empty(spec_verify_lmhead_workspace_bytes(B, K1 - 1, d, c.W.shape[1]),
                         dtype=torch.uint8, device=device)
        for i in range(n):
            spec_verify_lmhead(c.hidden, c.W, c.draft, c.tokens, c.temperature, seed=i, workspace=ws)
    else:
        props = torch.cuda.get_device_properties(device)
        l2 = int(getattr(props, "L2_cache_size", 0) or 129 * 2**20)
        name = args.profile.replace("-alone", "")
        sets, _ = workload_sets(name, device, l2)
        for i in range(n):
            c = sets[i % len(sets)]
            spec_verify_ex(c.target, c.draft, c.tokens, c.temperature, modes=uniform_mode(c.modes),
                           seed=i, overlap_previous=not args.profile.endswith("-alone"))
    torch.cuda.synchronize()
    print(f"profile run: {args.profile}, {n} steps", flush=True)


# ----------------------------------------------------------------- main


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="c4", choices=["c1", "c2", "c3", "c4"])
    ap.add_argument("--also", default="c2,c3,c4,c5,ragged,tree,lookup,commit",
                    help="other workloads reported as sub-results")
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--profile", choices=["c1", "c2", "c3", "c4", "c5", "c2-alone", "c3-alone", "c4-alone"],
                    help="run warmup+steps calls of one workload for ncu; no bench line")
    args = ap.parse_args()
    args.also = [a for a in args.also.split(",") if a]
    args.warmup = max(3, args.warmup)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if args.profile:
        profile_run(args, device)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)
    result = run_ours(args, rank, world, device)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
