#!/usr/bin/env python3
"""Benchmark of the batched speculative-sampling verification step on GB300.

One step = one spec_verify call over one batch of the workload (every row of
the batch normalised, alpha for every position, acceptance, first rejection,
residual/bonus draw).  Default workload: B=256, gamma=7, V=128256, bf16
logits, T=1, top-k 50 then top-p 0.9 (the 128k-vocabulary configuration the
throughput target is stated on).  Metric: verified draft positions per second
(sum_b gamma_b per call / call time), with the achieved HBM GB/s of the
dominant kernel against the measured copy bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Multi-GPU (under torchrun): every rank verifies its own batch (weak scaling;
sequences are independent, so no collective touches the data path); the
reported time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified draft positions/sec and achieved HBM GB/s (% of GB300 peak), 1 GPU"
UNIT = "positions/s"
FALLBACK_HBM_GBS = 6800.0
# kernels one spec_verify call launches: plan, select (streaming top-k), combine,
# the whole-row kernel of rows without top-k and its per-unit tail, and the
# dense cluster kernel (a kernel whose path no row takes exits at once);
# spec_verify_gumbel adds its one-pass kernel of unfiltered rows
LAUNCHES_PER_STEP = 6


def launches_per_step(rule: str = "sampling") -> int:
    return LAUNCHES_PER_STEP + (1 if rule == "gumbel" else 0)
# sources of each kernel whose DRAM traffic profiles/traffic.json records: a
# record counts only while these files are unchanged since its capture
_CSRC = "speculative_decoding_verification_20_gb300/csrc/"
KERNEL_SOURCES = {
    "stream": tuple(_CSRC + f for f in ("sv_stream.cu", "sv_keys.cuh", "sv_internal.cuh", "sv_finalize.cuh")),
    "free": tuple(_CSRC + f for f in ("sv_free.cu", "sv_cf.cuh", "sv_warp_sort.cuh", "sv_internal.cuh",
                                      "sv_finalize.cuh")),
    "gumbel": tuple(_CSRC + f for f in ("sv_gumbel.cu", "sv_internal.cuh", "sv_finalize.cuh")),
}


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_hash(path: str = "stream") -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[path]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# Issue peak of the SMs for an ALU-bound kernel: 152 SMs x 4 schedulers x one
# 32-thread instruction per cycle at the 2070 MHz maximum SM clock.
ALU_PEAK_TINST = 152 * 4 * 32 * 2.070e9 / 1e12


def recorded_instructions(rule: str, workload: str, path: str, default_batch: bool):
    """Thread instructions per launch of the dominant kernel (ncu
    smsp__thread_inst_executed.sum), from profiles/instructions.json; None for
    another batch size or kernel, or once its sources changed."""
    p = os.path.join(ROOT, "profiles", "instructions.json")
    try:
        with open(p) as f:
            rec = json.load(f).get(f"{rule}:{workload}")
    except Exception:
        return None
    if not default_batch or not rec or rec.get("path") != path or path not in KERNEL_SOURCES:
        return None
    if rec.get("kernel_hash") != kernel_hash(path):
        return None
    return rec.get("thread_inst_per_launch")


def recorded_traffic(workload: str, path: str, default_batch: bool):
    """DRAM bytes per launch of the dominant kernel at the workload's full size,
    from the committed ncu summary; None for another batch size, another
    kernel, or once that kernel's sources changed since the capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f).get(workload)
    except Exception:
        return None
    if not default_batch or not rec or path not in KERNEL_SOURCES or rec.get("path") != path:
        return None
    if rec.get("kernel_hash") != kernel_hash(path):
        return None
    return rec.get("bytes_per_launch")


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t_begin: float, t_end: float):
        rows = []
        for line in (self.out or "").splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        loaded = [s for s, _, _ in rows if s > 0]
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": max(m for _, m, _ in rows),
                "reasons": reasons, "samples": len(rows)}


def _cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def _oracle_rate(workload: str, threads: int, budget_s: float, seed0: int, max_batches: int = 256,
                 rule: str = "sampling"):
    """Positions per second of the fp64 oracle on whole sequences of the workload
    recipe, `threads` sequences at a time on `threads` host threads (rows are
    independent; the oracle is C called through ctypes, which releases the
    interpreter lock).  Inputs are built before each timed batch."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    from speculative_decoding_verification_20_gb300 import workloads

    oracle.build()

    def one(ni, b, seed):
        row = lambda x: None if x is None else x[b:b + 1]
        if rule == "gumbel":
            oracle.gumbel_verify(row(ni["target"]), row(ni["draft_tokens"]), row(ni["temperature"]),
                                 row(ni["num_draft"]), row(ni["top_k"]), row(ni["top_p"]), seed=seed)
        else:
            oracle.verify(row(ni["target"]), row(ni["draft"]), row(ni["draft_tokens"]), row(ni["temperature"]),
                          row(ni["num_draft"]), row(ni["top_k"]), row(ni["top_p"]), seed=seed)

    elapsed, positions, batches = 0.0, 0, 0
    with ThreadPoolExecutor(threads) as ex:
        while batches < max_batches and (batches == 0 or elapsed < budget_s):
            wl = workloads.make(workload, seed=seed0 + batches, B=threads)  # one sequence per thread
            ni = wl.numpy_inputs()
            t0 = time.perf_counter()
            list(ex.map(one, [ni] * threads, range(threads), [wl.seed] * threads))
            elapsed += time.perf_counter() - t0
            positions += wl.positions()
            batches += 1
    return positions / elapsed, batches * threads, positions, elapsed


def cpu_baseline(workload: str, budget_s: float = 10.0, rule: str = "sampling"):
    """The fp64 oracle, as it stands, on this host: one thread per core (rows are
    independent) and single-threaded, each on a bounded sample of whole
    sequences of the same workload recipe."""
    cores = os.cpu_count() or 1
    v1, n1, p1, e1 = _oracle_rate(workload, 1, budget_s, 10_000, rule=rule)
    vn, nn, pn, en = _oracle_rate(workload, cores, budget_s, 50_000, rule=rule)
    return {"value": vn, "unit": UNIT, "cores": cores, "kind": "oracle", "cpu_model": _cpu_model(),
            "single_thread_value": v1,
            "sample": f"{nn} whole sequences of the {workload} recipe ({pn} positions, {en:.1f} s wall on {cores} "
                      f"threads, one sequence per thread at a time); single-threaded: {n1} sequences "
                      f"({p1} positions, {e1:.1f} s)"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    cores = os.cpu_count() or 1
    times, positions = [], 0
    for step in range(args.warmup + args.steps):
        # each step: `cores` whole sequences of the workload, one per host thread
        v, n, pos, el = _oracle_rate(args.workload, cores, 0.0, 20_000 + step, max_batches=1, rule=args.rule)
        if step >= args.warmup:
            times.append(el)
            positions += pos
    total = sum(times)
    value = positions / total
    cfg = workload_config(args.workload)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / max(len(times), 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": cfg,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "cpu_model": _cpu_model(),
                             "sample": f"each step verifies {cores} whole sequences of the {args.workload} "
                                       f"recipe with the fp64 oracle, one per host thread"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def max_over_ranks(x: float, device=None) -> float:
    """The maximum of one float over all ranks (the slowest rank's time); x itself at world size 1."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, world: int, seconds_per_step: float) -> float:
    """Units of all ranks per second: every rank processes its own batch (weak scaling)."""
    return units_per_rank * world / seconds_per_step


def rank_seed(rank: int) -> int:
    """Each rank verifies its own synthetic batch: the workload seed is the rank."""
    return rank


def bytes_by_path(wl, stream_max_k: int, rule: str = "sampling") -> dict:
    """Algorithmic logit bytes each path of the library reads for this batch:
    greedy or 1 <= top_k <= stream_max_k rows stream (select kernel); rows with
    no top-k the whole-row kernel (free), except that shared noise on rows with
    no filter at all takes its one-pass kernel (gumbel); larger top-k the cluster
    kernel.  The sampling rule reads 2 gamma_b + 1 rows per sequence, shared
    noise the gamma_b + 1 target rows only."""
    import numpy as np

    gam = wl.gammas()
    T = wl.temperature.detach().cpu().numpy()
    k = np.zeros(wl.B, dtype=np.int64) if wl.top_k is None else wl.top_k.detach().cpu().numpy().astype(np.int64)
    k = np.where((k > 0) & (k < wl.V), k, 0)
    P = np.ones(wl.B) if wl.top_p is None else wl.top_p.detach().cpu().numpy().astype(np.float64)
    stream = (T == 0) | ((k >= 1) & (k <= stream_max_k))
    free = ~stream & (k == 0)
    gumbel = free & (P >= 1.0) if rule == "gumbel" else np.zeros(wl.B, dtype=bool)
    free &= ~gumbel
    es = 2 if wl.dtype == "bf16" else 4
    rowb = ((gam + 1) if rule == "gumbel" else (2 * gam + 1)) * wl.V * es
    out = {"stream": int(rowb[stream].sum()), "free": int(rowb[free].sum()),
           "dense": int(rowb[~stream & ~free & ~gumbel].sum())}
    if rule == "gumbel":
        out["gumbel"] = int(rowb[gumbel].sum())
    return out


def workload_config(name: str, B: int | None = None) -> dict:
    from speculative_decoding_verification_20_gb300.workloads import CONFIGS

    c = dict(CONFIGS[name])
    if B is not None:
        c["B"] = B
    filt = {"v128k": "T=1, top-k 50 then top-p 0.9", "v32k": "T=0.8, no filter", "b1024": "T=1, no filter",
            "tiny": "T=1, no filter", "ragged": "T in {0,.3,.7,1,1.2}, top-p U[.8,1]"}[name]
    return {"workload": f"{name}: B={c['B']}, gamma={c['G']}{' (ragged 1..8)' if name == 'ragged' else ''}, "
                        f"V={c['V']}, {c['dtype']} logits, {filt}",
            "B": c["B"], "gamma": c["G"], "V": c["V"], "logits": c["dtype"]}


def run_kseq(args, sv, workloads, world, rank, dev):
    """K-SEQ: one position per row with k candidates.  Rows with top-k <= 256 take the
    streaming select kernel and solve rho* over their kept lists in the combine
    kernel; the others are held on chip by the cluster kernel while it finds rho*.
    Positions = rows."""
    import torch
    import torch.distributed as dist

    wl = workloads.make_kseq(args.workload, seed=rank_seed(rank), device=dev, B=args.batch)
    B, K, V = wl.B, wl.K, wl.V
    dt = sv.SV_BF16 if wl.dtype == "bf16" else sv.SV_F32
    ws = torch.empty(max(int(sv.load_library().spec_verify_kseq_workspace_size(B, K, V, dt)), 256), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(seed, events=None):
        return sv.spec_verify_kseq(wl.target, wl.draft, wl.candidates, wl.temperature, wl.num_candidates, wl.top_k,
                                   wl.top_p, seed=seed, workspace=ws, events=events)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    graphs = []
    left, seed = args.steps, 1_000_000
    while left > 0 and not args.eager:
        n = min(100, left)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n):
                step(seed + i)
        graphs.append(g)
        seed += n
        left -= n
    for g in graphs:
        g.replay()
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    props = torch.cuda.get_device_properties(dev)
    smi_id = f"GPU-{props.uuid}" if getattr(props, "uuid", None) else str(int(os.environ.get("LOCAL_RANK", "0")))
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(smi_id) as clk:
        wall0 = time.perf_counter()
        t0.record(stream)
        if graphs:
            for g in graphs:
                g.replay()
        else:
            for i in range(args.steps):
                step(1_000_000 + i)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        wall1 = time.perf_counter()
    ms_step = max_over_ranks(t0.elapsed_time(t1), dev) / args.steps
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a_, b_ in kev:
        a_.record(stream)
        b_.record(stream)
    torch.cuda.synchronize(dev)
    tk = None if wl.top_k is None else wl.top_k.detach().cpu()
    listed = tk is not None and bool(((tk >= 1) & (tk <= sv.SV_STREAM_MAX_TOP_K)).all())
    main = "stream" if listed else "dense"  # the kernel that reads this batch's logits
    for i in range(args.steps):
        step(3_000_000 + i, events={main: kev[i]})
    torch.cuda.synchronize(dev)
    kernel_ms = sum(a.elapsed_time(b) for a, b in kev) / args.steps
    peak, peak_kind = measured_peak()
    nbytes = wl.logit_bytes()
    value = whole_job_rate(wl.positions(), world, ms_step * 1e-3)
    if rank != 0:
        return 0
    achieved = nbytes / (kernel_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "timed_region": ("K calls replayed from CUDA graphs of up to 100 captured calls"
                                                 if graphs else "K calls issued one by one"),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": f"{args.workload}: B={B} rows (one position each), K={K} candidates, V={V}, "
                               f"{wl.dtype} logits", "rule": "kseq", "B": B, "K": K, "V": V, "logits": wl.dtype,
                   "l2": "%.0f MB of logits per step vs 129 MB L2" % (nbytes / 1e6)},
        "hbm_gbs_step": nbytes / (ms_step * 1e-3) / 1e9, "hbm_frac_step": nbytes / (ms_step * 1e-3) / 1e9 / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     "kernel": ("select_kernel (streaming top-k path; K-SEQ on the kept lists in combine)"
                                if main == "stream" else "dense_kernel (cluster path, K-SEQ)"),
                     "kernel_ms": kernel_ms,
                     "algorithmic_bytes_per_launch": nbytes, "traffic": None},
        "e2e": None, "gpu_launches": LAUNCHES_PER_STEP * args.steps, "clocks": clk.summary(wall0, wall1),
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="v128k")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--batch", type=int, default=None, help="override B (profiling of smaller cases)")
    ap.add_argument("--eager", action="store_true", help="time calls issued one by one (no CUDA graph)")
    ap.add_argument("--rule", default="sampling", choices=["sampling", "gumbel", "kseq"],
                    help="verification rule: speculative sampling (spec_verify), shared noise "
                         "(spec_verify_gumbel) or K-SEQ candidates at one position (spec_verify_kseq; "
                         "workloads kseq32k, kseq128k)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist

    import speculative_decoding_verification_20_gb300 as sv
    from speculative_decoding_verification_20_gb300 import _build, workloads

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        _build.build()
    if world > 1:
        dist.barrier()
    sv.load_library()

    if args.rule == "kseq":
        return run_kseq(args, sv, workloads, world, rank, dev)
    wl = workloads.make(args.workload, seed=rank_seed(rank), device=dev, B=args.batch)
    B, G, V = wl.B, wl.G, wl.V
    stream = torch.cuda.current_stream(dev)
    ws = torch.empty(sv.workspace_size(B, G, V, sv.SV_BF16 if wl.dtype == "bf16" else sv.SV_F32), dtype=torch.uint8,
                     device=dev)

    def step(seed, events=None):
        if args.rule == "gumbel":
            return sv.spec_verify_gumbel(wl.target, wl.draft_tokens, wl.temperature, wl.num_draft, wl.top_k,
                                         wl.top_p, seed=seed, workspace=ws, events=events)
        return sv.spec_verify(wl.target, wl.draft, wl.draft_tokens, wl.temperature, wl.num_draft, wl.top_k, wl.top_p,
                              seed=seed, workspace=ws, events=events)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)

    # the dominant kernel: the path that reads the most logits
    path_bytes = bytes_by_path(wl, sv.SV_STREAM_MAX_TOP_K, args.rule)
    main = max(path_bytes, key=path_bytes.get)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    props = torch.cuda.get_device_properties(dev)
    smi_id = f"GPU-{props.uuid}" if getattr(props, "uuid", None) else str(local)
    # The timed region replays the K calls from CUDA graphs captured once (up to
    # 100 calls each, every call with its own seed), as a decode loop issues its
    # steps: the device time of the library's own kernels, without the Python
    # binding's per-call host overhead (which bounds small batches when the
    # calls are issued one by one; that eager figure is reported beside it).
    graphs = []
    if not args.eager:
        left, seed = args.steps, 1_000_000
        while left > 0:
            n = min(100, left)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for i in range(n):
                    step(seed + i)
            graphs.append(g)
            seed += n
            left -= n
        for g in graphs:  # one untimed replay of each graph
            g.replay()
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(smi_id) as clk:
        wall0 = time.perf_counter()
        # the timed region: K production steps back to back, nothing recorded
        # between the call's kernels (their programmatic dependent launches overlap)
        t0.record(stream)
        if graphs:
            for g in graphs:
                g.replay()
        else:
            for i in range(args.steps):
                step(1_000_000 + i)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        wall1 = time.perf_counter()
    if world > 1:
        dist.barrier()
    ms_total = max_over_ranks(t0.elapsed_time(t1), dev)
    ms_step = ms_total / args.steps
    # the same K calls issued one by one from Python (host launch overhead included)
    q0, q1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    q0.record(stream)
    for i in range(args.steps):
        step(2_000_000 + i)
    q1.record(stream)
    torch.cuda.synchronize(dev)
    ms_step_eager = max_over_ranks(q0.elapsed_time(q1), dev) / args.steps
    positions = wl.positions()
    value = whole_job_rate(positions, world, ms_step * 1e-3)

    # the dominant kernel's own duration: a second run of K steps in which the
    # library records CUDA events on the launching stream around that kernel
    # (an event between two kernels of the call serialises them, so this run
    # is kept apart from the timed region above)
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a_, b_ in kev:  # torch creates the underlying CUDA events on their first record
        a_.record(stream)
        b_.record(stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for i in range(args.steps):
        step(3_000_000 + i, events={main: kev[i]})
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms_step_with_events = e0.elapsed_time(e1) / args.steps
    kernel_ms = [a.elapsed_time(b) for a, b in kev]
    kernel_ms_avg = sum(kernel_ms) / len(kernel_ms)
    bytes_per_launch = sum(path_bytes.values())
    main_bytes = path_bytes[main]
    achieved = main_bytes / (kernel_ms_avg * 1e-3) / 1e9
    peak, peak_kind = measured_peak()

    # end to end through the host-buffer entry point: pinned inputs in, results out, every step
    e2e = None
    if args.e2e_steps > 0 and args.rule == "gumbel":
        # end to end through the Python API: pinned inputs copied in, results copied out
        pin = lambda x: None if x is None else x.detach().cpu().contiguous().pin_memory()
        h = [pin(x) for x in (wl.target, wl.draft_tokens, wl.temperature, wl.num_draft, wl.top_k, wl.top_p)]
        dbuf = [None if x is None else torch.empty_like(x, device=dev) for x in h]
        hout = [torch.empty(B, dtype=torch.int32).pin_memory(), torch.empty(B, G + 1, dtype=torch.int32).pin_memory()]

        def e2e_step(seed):
            for d, x in zip(dbuf, h):
                if x is not None:
                    d.copy_(x, non_blocking=True)
            r = sv.spec_verify_gumbel(dbuf[0], dbuf[1], dbuf[2], dbuf[3], dbuf[4], dbuf[5], seed=seed, workspace=ws)
            hout[0].copy_(r["accepted_len"], non_blocking=True)
            hout[1].copy_(r["out_tokens"], non_blocking=True)
            torch.cuda.current_stream(dev).synchronize()

        for i in range(3):
            e2e_step(i)
        if world > 1:
            dist.barrier()
        w0 = time.perf_counter()
        for i in range(args.e2e_steps):
            e2e_step(2_000_000 + i)
        w1 = time.perf_counter()
        e_step = max_over_ranks(w1 - w0, dev) / args.e2e_steps
        e2e = {"value": whole_job_rate(positions, world, e_step), "unit": UNIT,
               "h2d_bytes_per_step": sum(x.numel() * x.element_size() for x in h if x is not None),
               "d2h_bytes_per_step": sum(x.numel() * x.element_size() for x in hout), "steps": args.e2e_steps,
               "ms_per_step": e_step * 1e3}
    elif args.e2e_steps > 0:
        pin = lambda x: None if x is None else x.detach().cpu().contiguous().pin_memory()
        h = [pin(x) for x in (wl.target, wl.draft, wl.draft_tokens, wl.temperature, wl.num_draft, wl.top_k,
                               wl.top_p)]
        staging = torch.empty(sv.host_staging_size(B, G, V, sv.SV_BF16 if wl.dtype == "bf16" else sv.SV_F32,
                                                   h[4] is not None, h[5] is not None, h[6] is not None),
                              dtype=torch.uint8, device=dev)
        outs = None
        for i in range(3):
            outs = sv.spec_verify_host(*h, seed=i, staging=staging, outputs=outs)
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        w0 = time.perf_counter()
        for i in range(args.e2e_steps):
            outs = sv.spec_verify_host(*h, seed=2_000_000 + i, staging=staging, outputs=outs)
        w1 = time.perf_counter()
        e_step = max_over_ranks(w1 - w0, dev) / args.e2e_steps
        h2d = sum(x.numel() * x.element_size() for x in h if x is not None)
        d2h = sum(x.numel() * x.element_size() for x in outs.values())
        e2e = {"value": whole_job_rate(positions, world, e_step), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": args.e2e_steps, "ms_per_step": e_step * 1e3}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0
    clocks = clk.summary(wall0, wall1)
    traffic = recorded_traffic(args.workload, main, args.batch is None) if args.rule == "sampling" else None
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_source": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                else "fallback 6.8 TB/s",
                "kernel": {"stream": "select_kernel (streaming top-k path)",
                           "free": "free_kernel (whole-row path: rows without top-k)",
                           "dense": "dense_kernel (cluster path)",
                           "gumbel": "gumbel_kernel (one pass of shared noise: rows without filters)"}[main],
                "kernel_ms": kernel_ms_avg, "algorithmic_bytes_per_launch": main_bytes,
                "traffic": traffic,
                "timing": "kernel events in a separate run of K steps "
                          f"({ms_step_with_events:.4f} ms per step with the events recorded)"}
    if args.rule == "gumbel" and main in ("free", "gumbel"):
        # shared noise on rows without top-k: a quarter Philox block and the noise test
        # per token make the kernel issue-bound, not HBM-bound
        inst = recorded_instructions(args.rule, args.workload, main, args.batch is None)
        hbm = dict(roofline)
        roofline = {"bound": "alu", "unit": "T thread-inst/s", "peak": ALU_PEAK_TINST,
                    "peak_source": "152 SMs x 4 schedulers x 32 threads x 2070 MHz (one instruction per scheduler "
                                   "per cycle)",
                    "achieved": None if inst is None else inst / (kernel_ms_avg * 1e-3) / 1e12,
                    "thread_inst_per_launch": inst, "kernel": hbm["kernel"], "kernel_ms": kernel_ms_avg,
                    "hbm": {"achieved_gbs": achieved, "frac": achieved / peak, "peak": peak}, "traffic": None,
                    "timing": hbm["timing"]}
        roofline["frac"] = None if inst is None else roofline["achieved"] / ALU_PEAK_TINST
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "ms_per_step_eager": ms_step_eager,
        "timed_region": ("K calls replayed from CUDA graphs of up to 100 captured calls" if graphs
                         else "K calls issued one by one"),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": wl.dtype, "data": "synthetic",
        "config": dict(workload_config(args.workload, B), rule=args.rule,
                       l2="inputs larger than L2: %.0f MB of logits per step vs 129 MB L2" % (bytes_per_launch / 1e6),
                       parallelism=f"replicas x{world} (independent batches per GPU)"),
        "hbm_gbs_step": bytes_per_launch / (ms_step * 1e-3) / 1e9,
        "hbm_frac_step": bytes_per_launch / (ms_step * 1e-3) / 1e9 / peak,
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": launches_per_step(args.rule) * args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(args.workload, rule=args.rule)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
