"""Benchmark of the chunkwise Gated DeltaNet forward on one GB300 (or N replicas).

One step = one gdn_chunk_fwd over the whole workload (every step of the hot
path: gate cumsum, decayed Gram, triangular solve, WY factors, the serial state
pass and the outputs), inputs resident in HBM.  L2 is flushed (a 512 MiB write)
between timed steps; each step is timed with CUDA events on the launching
stream.  Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-cpu-baseline]

--impl reference times the fp64 CPU oracle (the only other implementation of
this path) on the host cores, each step a bounded sample of the workload.
Under torchrun (N > 1) every rank runs its own replica of the workload (no
collective on the data path); rank 0 prints.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "gated-DeltaNet chunkwise fwd tokens/s and % of roofline, 1×GB300"
LINEAR_METRIC = "linear-attention (Mamba2 gate) chunkwise fwd tokens/s and % of roofline, 1×GB300"
BWD_METRIC = "gated-DeltaNet backward tokens/s and % of roofline, 1×GB300"
DECODE_METRIC = "gated-DeltaNet decode step tokens/s and % of roofline, 1×GB300"
L2_FLUSH_BYTES = 512 << 20


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, source="fallback")


def algorithmic(inp: dict) -> dict:
    """Algorithmic bytes and FLOPs of one forward.

    Bytes: q, k, v read and out written once in the qkv dtype, log_alpha and
    beta read once (fp32), S0 read and S_final written once (fp32 dv x dk per
    (sequence, head)).  FLOPs: the dense chunk tiles per token and head,
    2C(3dk + 2dv) + 6 dk dv (Gram K K^T and Q K^T, W~ and U, delta, Q S^T,
    P delta and the state update)."""
    esz = 2 if inp["dtype"] == "bf16" else 4
    th = inp["B"] * inp["T"] * inp["H"]
    dk, dv, C = inp["dk"], inp["dv"], inp["C"]
    units = inp["N"] * inp["H"]
    gates = 4 if inp.get("linear") else 8  # the linear mode reads no beta
    by = th * ((2 * dk + dv) * esz + dv * esz + gates)
    if inp["S0"] is not None:
        by += units * dv * dk * 4
    by += units * dv * dk * 4  # S_final
    fl = th * (2 * C * (3 * dk + 2 * dv) + 6 * dk * dv)
    return dict(bytes=by, flops=fl, tok_heads=th)


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        if not self.lines:
            return None
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        loaded = [s for s in sm if s >= 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, dev) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def cpu_oracle_time(inp: dict, budget_s: float = 20.0):
    """Time the fp64 oracle on the host cores over a bounded sample of
    (sequence, head) units of the workload.  Returns (tokens/s, cores, sample).
    The linear mode runs the oracle with erase strength 0 and write strength 1."""
    from oracle import native
    ew = {}
    beta = inp["beta"]
    if inp.get("linear"):
        beta = torch.zeros_like(inp["log_alpha"])  # unused once erase and write are given
        ew = dict(erase=beta, write=torch.ones_like(inp["log_alpha"]))
    spans = native.spans(inp["B"], inp["T"], inp["cu_seqlens"])
    H = inp["H"]
    units_all = [(s, h) for s in range(len(spans)) for h in range(H)]
    cores = native.max_threads()
    # probe one unit to size the sample
    probe = [units_all[0]]
    t0 = time.perf_counter()
    native.gdn_units_c(inp["q"], inp["k"], inp["v"], inp["log_alpha"], beta, inp["S0"],
                       inp["cu_seqlens"], probe, n_threads=1, **ew)
    per_tok_thread = (time.perf_counter() - t0) / max(1, spans[0][1])
    total_tok_heads = sum(l for _, l in spans) * H
    est = per_tok_thread * total_tok_heads / max(1, cores)
    if est <= budget_s:
        units = units_all
    else:
        frac = budget_s / est
        step = max(1, int(round(1 / frac)))
        units = units_all[::step]
    t0 = time.perf_counter()
    native.gdn_units_c(inp["q"], inp["k"], inp["v"], inp["log_alpha"], beta, inp["S0"],
                       inp["cu_seqlens"], units, n_threads=cores, **ew)
    dt = time.perf_counter() - t0
    tok_heads = sum(spans[s][1] for s, _ in units)
    tokens_per_s = tok_heads / H / dt  # tokens of all heads, per second
    sample = (f"{len(units)} of {len(units_all)} (sequence, head) units of the workload "
              f"({tok_heads} token-heads), fp64 per-token recurrence, OpenMP over units")
    return tokens_per_s, cores, sample, dt


def run_reference(args, w, world, rank):
    if rank != 0:
        return
    inp = dict(workloads.make_inputs(w), linear=w.linear)
    for _ in range(args.warmup if args.warmup > 0 else 0):
        pass  # the oracle has no state to warm; warm-up steps are not timed
    vals, times = [], []
    cores = sample = None
    for _ in range(args.steps):
        v, cores, sample, dt = cpu_oracle_time(inp, budget_s=args.ref_budget)
        vals.append(v)
        times.append(dt)
    value = statistics.median(vals)
    line = {"metric": LINEAR_METRIC if w.linear else METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * n_tokens_of(inp) / value, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": w.name, "B": inp["B"], "H": inp["H"], "T": inp["T"],
                       "dk": w.dk, "dv": w.dv, "C": w.C},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def measured_traffic(workload: str):
    """DRAM bytes per launch of the workload's dominant kernel from its recorded ncu
    capture (profiles/dram_traffic.json), or None when there is none or the kernel's
    source has changed since the capture (its SHA-256 differs)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        rec = json.load(open(path))["workloads"][workload]
        src = open(os.path.join(ROOT, rec["source"]), "rb").read()
    except (OSError, KeyError, ValueError):
        return None
    if hashlib.sha256(src).hexdigest() != rec["source_sha256"]:
        return None
    return rec["dram_read_bytes"] + rec["dram_write_bytes"]


def decode_algorithmic(inp: dict) -> dict:
    """Algorithmic bytes and FLOPs of one decode step over the batch: the state read
    and written once (fp32 dv x dk per (sequence, head)), q, k, v read and out
    written once in the qkv dtype, log_alpha and beta read once.  FLOPs: S k and
    S q (4 dk dv), the rank-one update (3 dk dv), per (sequence, head)."""
    esz = 2 if inp["dtype"] == "bf16" else 4
    units = inp["N"] * inp["H"]
    dk, dv = inp["dk"], inp["dv"]
    by = units * (2 * dk * dv * 4 + (2 * dk + dv) * esz + dv * esz + 8)
    return dict(bytes=by, flops=units * 7 * dk * dv)


def decode_oracle_time(inp: dict):
    """Time the fp64 oracle for one decode step of every (sequence, head) on the host
    cores.  Returns (tokens/s, cores, sample, seconds)."""
    from oracle import native
    cores = native.max_threads()
    q, k, v = (inp[n].unsqueeze(1) for n in ("q", "k", "v"))
    la, be = inp["log_alpha"].unsqueeze(1), inp["beta"].unsqueeze(1)
    units = [(s, h) for s in range(inp["N"]) for h in range(inp["H"])]
    t0 = time.perf_counter()
    native.gdn_units_c(q, k, v, la, be, inp["S"], None, units, n_threads=cores)
    dt = time.perf_counter() - t0
    sample = (f"all {len(units)} (sequence, head) units, one token each, fp64 recurrence step, "
              f"OpenMP over units")
    return inp["N"] / dt, cores, sample, dt


def run_decode(args, w, world, rank, local):
    """The decode workloads: one step = one gdn_decode_step over the whole batch."""
    if args.impl == "reference":
        if rank != 0:
            return
        inp = workloads.make_decode_inputs(w)
        vals, cores, sample = [], None, None
        for _ in range(args.steps):
            v, cores, sample, _ = decode_oracle_time(inp)
            vals.append(v)
        value = statistics.median(vals)
        print(json.dumps({
            "metric": DECODE_METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * inp["N"] / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": w.name, "N": inp["N"], "H": inp["H"], "dk": w.dk, "dv": w.dv},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}), flush=True)
        return
    import chunkwise_gated_deltanet_gb300 as gdn
    gdn.load_library()
    assert torch.cuda.is_available(), "bench.py needs a CUDA device"
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inp = workloads.make_decode_inputs(w)
    d = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in inp.items()}
    N, H = inp["N"], inp["H"]
    out = torch.empty(d["v"].shape, dtype=d["v"].dtype, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():  # the state evolves in place from step to step, as in decoding
        gdn.gdn_decode_step(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["S"], out,
                            stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
        flush.zero_()
    torch.cuda.synchronize()
    gdn.gdn_check_status(stream)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        t_wall0 = time.perf_counter()
        for i in range(args.steps):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
            flush.zero_()
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
    barrier(world)
    gdn.gdn_check_status(stream)
    ms = max_over_ranks(sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / args.steps,
                        world, dev)
    alg = decode_algorithmic(inp)
    peaks = load_peaks()
    sec = ms * 1e-3
    achieved_gbs = alg["bytes"] / sec / 1e9
    tokens = N * world

    # end to end through the public call: the token's inputs and the state go in from
    # pinned host memory, the outputs and the state come back
    host_in = {k: inp[k].pin_memory() for k in ("q", "k", "v", "log_alpha", "beta", "S")}
    out_h = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    S_h = torch.empty(inp["S"].shape, dtype=torch.float32, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = out_h.numel() * out_h.element_size() + S_h.numel() * S_h.element_size()

    def e2e_step():
        # the public call on pinned host tensors: the token's inputs and the state go in,
        # the output and the new state come back (copies pipelined over slices of
        # sequences); it returns with both written
        return gdn.decode_step(host_in["q"], host_in["k"], host_in["v"], host_in["log_alpha"],
                               host_in["beta"], host_in["S"])

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    t_e2e = time.perf_counter()
    for _ in range(args.e2e_steps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks((time.perf_counter() - t_e2e) * 1e3 / args.e2e_steps, world, dev)
    gdn.gdn_check_status(stream)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, sample, _ = decode_oracle_time(inp)
        cpu = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps({
            "metric": DECODE_METRIC, "value": tokens / sec, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "N": N, "H": H, "dk": w.dk, "dv": w.dv,
                       "qkv_dtype": w.dtype, "state": "fp32, updated in place",
                       "l2": "flushed between timed steps (512 MiB write)",
                       "parallelism": f"replicas{world}"},
            "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": achieved_gbs / peaks["hbm_gbs"],
                         "traffic": measured_traffic(w.name), "peak_source": peaks["source"],
                         "algorithmic_bytes": alg["bytes"]},
            "clocks": clk.summary(),
            "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "timing": "host clock around the synchronous public call decode_step on "
                              "pinned host tensors (copies pipelined over 4 slices)"},
            "gpu_launches": args.steps,
            "cpu_baseline": cpu,
            "wall_s_timed_region": t_wall}), flush=True)


def run_seqpar(args, w, world, rank, local):
    """The sequence-parallel split of one workload over R = --seqpar ranks, with every
    rank's work timed alone on this one GPU: phase 1 (rank 0's segment from S0; a
    middle rank's (M, L) passes on two streams), then phase 2 (the fold and the
    segment from the folded start state; in the linear mode at bf16 d = 128 the ranks
    r > 0 run their segment from zero in phase 1 and only correct it in phase 2).  The critical path max(phase 1) +
    max(phase 2) is what R GPUs would take, less the exchange of two state-sized
    tensors per rank, which is not timed here."""
    import chunkwise_gated_deltanet_gb300 as gdn
    from chunkwise_gated_deltanet_gb300 import seqpar
    if world != 1 or w.varlen:
        raise SystemExit("--seqpar times R ranks on one GPU, for fixed-length workloads")
    gdn.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inp = workloads.make_inputs(w)
    d = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in inp.items()}
    Rk, C, T = args.seqpar, w.C, inp["T"]
    ops = seqpar.cuda_ops()
    bounds = seqpar.segment_bounds(T, Rk, C)
    names = ("q", "k", "v", "log_alpha", "beta")
    segs = [[seqpar.segment(d[n], b) for n in names] for b in bounds]
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def timed(fn):
        flush.zero_()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        res = fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1), res

    un, p1, p2 = [], [[] for _ in range(Rk)], [[] for _ in range(Rk)]
    for it in range(max(3, args.warmup) + args.steps):
        keep = it >= max(3, args.warmup)
        t, _ = timed(lambda: ops.forward(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                         d["S0"], C, w.linear))
        if keep:
            un.append(t)
        first = []
        for r in range(Rk):
            t, res = timed(lambda r=r: seqpar.phase1(r, Rk, *segs[r], d["S0"], C, w.linear, ops))
            first.append(res)
            if keep:
                p1[r].append(t)
        Ms = torch.stack([m for m, _, _ in first])
        Ls = torch.stack([l for _, l, _ in first])
        for r in range(Rk):
            t, _ = timed(lambda r=r: seqpar.phase2(r, *segs[r], C, w.linear, ops, Ms, Ls,
                                                   first[r][2]))
            if keep:
                p2[r].append(t)
    gdn.gdn_check_status()
    med = statistics.median
    ph1 = [med(x) for x in p1]
    ph2 = [med(x) for x in p2]
    crit = max(ph1) + max(ph2)
    tokens = inp["B"] * T
    print(json.dumps({
        "metric": ("linear-attention (Mamba2 gate)" if w.linear else "gated-DeltaNet") +
                  f" sequence-parallel fwd tokens/s over {Rk} ranks "
                  "(per-rank work timed on one GPU)",
        "value": tokens / (crit * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": crit, "higher_is_better": True,
        "scaling": "strong", "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "ranks": Rk, "segments": bounds,
                   "l2": "flushed before every timed phase",
                   "timing": "each rank's phase timed alone with CUDA events (host launch "
                             "overhead included); exchange not timed"},
        "unsplit_ms": med(un), "speedup_vs_unsplit": med(un) / crit,
        "phase1_ms": ph1, "phase2_ms": ph2}), flush=True)


def bwd_algorithmic(inp: dict) -> dict:
    """Algorithmic bytes and FLOPs of one backward.  Bytes: q, k, v, d_out read and
    d_q, d_k, d_v written once in the qkv dtype; log_alpha, beta read and their
    gradients written once (fp32); S0 / dS_final read and d_S0 written once when
    present.  FLOPs per token and head: the forward state step p = S k and
    S <- a S + u k^T (5 dk dv) and the reverse step G += dO q^T, dq, du = G k,
    <G, S>, dk and G <- a G + dp k^T (17 dk dv)."""
    esz = 2 if inp["dtype"] == "bf16" else 4
    th = inp["B"] * inp["T"] * inp["H"]
    dk, dv = inp["dk"], inp["dv"]
    units = inp["N"] * inp["H"]
    by = th * (2 * (2 * dk + dv) * esz + 16)
    state = units * dv * dk * 4
    by += state * ((inp["S0"] is not None) + 2)  # S0, dS_final, d_S0
    return dict(bytes=by, flops=th * 22 * dk * dv)


def run_bwd(args, w, world, rank, local):
    """One step = one gdn_chunk_bwd over the workload, on the path --bwd-path names."""
    if args.impl == "reference":
        if rank != 0:
            return
        inp = workloads.make_inputs(w)
        grads = workloads.make_grad_inputs(inp)
        vals, cores, sample = [], None, None
        for _ in range(args.steps):
            v, cores, sample, _ = bwd_oracle_time(inp, grads, args.ref_budget)
            vals.append(v)
        value = statistics.median(vals)
        print(json.dumps({
            "metric": BWD_METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * inp["B"] * inp["T"] / value, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference", "config": {"workload": w.name, "pass": "backward"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}), flush=True)
        return
    import chunkwise_gated_deltanet_gb300 as gdn
    gdn.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inp = workloads.make_inputs(w)
    grads = workloads.make_grad_inputs(inp)
    d = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in inp.items()}
    gd = {k: v.to(dev) for k, v in grads.items()}
    B, T, H, dk, dv, N = inp["B"], inp["T"], inp["H"], w.dk, w.dv, inp["N"]
    outs = [torch.empty_like(d["q"]), torch.empty_like(d["k"]), torch.empty_like(d["v"]),
            torch.empty_like(d["log_alpha"]), torch.empty_like(d["beta"]),
            torch.empty((N, H, dv, dk), dtype=torch.float32, device=dev)]
    nbytes = gdn.gdn_chunk_bwd_workspace_bytes(B, H, T, dk, dv, N)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    path = {"auto": gdn.GDN_BWD_AUTO, "tokens": gdn.GDN_BWD_TOKENS,
            "chunked": gdn.GDN_BWD_CHUNKED}[args.bwd_path]
    taken = gdn.gdn_bwd_select_path(dk, dv, inp["q"].dtype) if path == gdn.GDN_BWD_AUTO else path
    launches = 25 if taken == gdn.GDN_BWD_CHUNKED and B * T > 0 else 2

    def step():
        gdn.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["S0"],
                          gd["d_out"], gd["dS_final"], *outs, ws, d["cu_seqlens"], stream=stream,
                          path=path)

    for _ in range(max(3, args.warmup)):
        step()
        flush.zero_()
    torch.cuda.synchronize()
    gdn.gdn_check_status(stream)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        t_wall0 = time.perf_counter()
        for i in range(args.steps):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
            flush.zero_()
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
    barrier(world)
    gdn.gdn_check_status(stream)
    ms = max_over_ranks(sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / args.steps,
                        world, dev)
    alg = bwd_algorithmic(dict(inp, dk=dk, dv=dv))
    peaks = load_peaks()
    sec = ms * 1e-3
    tokens = B * T * world
    # fp32 CUDA-core peak: 152 SMs x 128 FMA lanes x 2 FLOP x the maximum SM clock
    alu_peak = 152 * 128 * 2 * 2.07e9 / 1e12
    achieved_tf = alg["flops"] / sec / 1e12

    host_in = {k: (inp[k].pin_memory() if inp[k] is not None else None)
               for k in ("q", "k", "v", "log_alpha", "beta", "S0", "cu_seqlens")}
    host_g = {k: v.pin_memory() for k, v in grads.items()}
    host_out = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
    h2d = sum(t.numel() * t.element_size() for t in list(host_in.values()) + list(host_g.values())
              if t is not None)
    d2h = sum(t.numel() * t.element_size() for t in host_out)

    def e2e_step():
        for key, t in host_in.items():
            if t is not None:
                d[key].copy_(t, non_blocking=True)
        for key, t in host_g.items():
            gd[key].copy_(t, non_blocking=True)
        step()
        for ho, o in zip(host_out, outs):
            ho.copy_(o, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, world, dev)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, sample, _ = bwd_oracle_time(inp, grads, args.ref_budget)
        cpu = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps({
            "metric": BWD_METRIC, "value": tokens / sec, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": w.name, "pass": "backward", "B": B, "H": H, "T": T,
                       "dk": dk, "dv": dv, "qkv_dtype": w.dtype, "workspace_bytes": nbytes,
                       "path": "chunked" if taken == gdn.GDN_BWD_CHUNKED else "tokens",
                       "l2": "flushed between timed steps (512 MiB write)",
                       "parallelism": f"replicas{world}"},
            "roofline": {"bound": "alu", "achieved": achieved_tf, "peak": alu_peak,
                         "unit": "TFLOP/s", "frac": achieved_tf / alu_peak, "traffic": None,
                         "peak_source": "derived: fp32 FMA lanes x 2 x max SM clock",
                         "algorithmic_flops": alg["flops"],
                         "hbm_gbs": alg["bytes"] / sec / 1e9,
                         "hbm_frac": alg["bytes"] / sec / 1e9 / peaks["hbm_gbs"]},
            "clocks": clk.summary(),
            "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": launches * args.steps,
            "cpu_baseline": cpu,
            "wall_s_timed_region": t_wall}), flush=True)


def bwd_oracle_time(inp: dict, grads: dict, budget_s: float = 20.0):
    """Time the fp64 backward oracle (numpy, one process) over a bounded sample of
    (sequence, head) units.  Returns (tokens/s, cores, sample, seconds)."""
    from oracle import backward as BW
    from oracle import native
    spans = native.spans(inp["B"], inp["T"], inp["cu_seqlens"])
    H = inp["H"]
    units = [(s, h) for s in range(len(spans)) for h in range(H)]
    arr = {k: inp[k].double().numpy() for k in ("q", "k", "v", "log_alpha", "beta")}
    dO = grads["d_out"].double().numpy()
    dSf = grads["dS_final"].double().numpy()
    S0 = None if inp["S0"] is None else inp["S0"].double().numpy()
    done, toks = 0, 0
    t0 = time.perf_counter()
    for s, h in units:
        r0, ln = spans[s]
        b, t_ = (0, r0) if inp["cu_seqlens"] is not None else (s, 0)
        sl = slice(t_, t_ + ln)
        BW.gdn_sequence_bwd(arr["q"][b, sl, h], arr["k"][b, sl, h], arr["v"][b, sl, h],
                            arr["log_alpha"][b, sl, h], arr["beta"][b, sl, h],
                            None if S0 is None else S0[s, h], dO[b, sl, h], dSf[s, h])
        done += 1
        toks += ln
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    sample = (f"{done} of {len(units)} (sequence, head) units ({toks} token-heads), fp64 "
              "per-token reverse recurrence, numpy, one process")
    return toks / H / dt, 1, sample, dt


def n_tokens_of(inp):
    return inp["B"] * inp["T"]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=workloads.HEADLINE,
                    choices=sorted(workloads.WORKLOADS) + sorted(workloads.DECODE_WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--ref-budget", type=float, default=20.0)
    ap.add_argument("--T", type=int, default=0,
                    help="override the tokens per sequence of a fixed-length workload "
                         "(for small profiling captures; the default is the workload's)")
    ap.add_argument("--bwd", action="store_true",
                    help="time the backward (gdn_chunk_bwd) of the workload instead")
    ap.add_argument("--bwd-path", choices=("auto", "tokens", "chunked"), default="auto",
                    help="backward kernel family (auto: the library's choice for the sizes)")
    ap.add_argument("--seqpar", type=int, default=0,
                    help="time the sequence-parallel split over this many ranks on one GPU")
    args = ap.parse_args()
    if args.T > 0:  # a smaller case of the same workload (profiling captures)
        import dataclasses
        base = workloads.WORKLOADS[args.workload]
        workloads.WORKLOADS[args.workload] = dataclasses.replace(base, T=args.T)
    world, rank, local = dist_setup()
    if args.seqpar > 0 and args.impl != "reference":
        run_seqpar(args, workloads.WORKLOADS[args.workload], world, rank, local)
        return
    if args.bwd:
        run_bwd(args, workloads.WORKLOADS[args.workload], world, rank, local)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    if args.workload in workloads.DECODE_WORKLOADS:
        run_decode(args, workloads.DECODE_WORKLOADS[args.workload], world, rank, local)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    w = workloads.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w, world, rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    import chunkwise_gated_deltanet_gb300 as gdn
    gdn.load_library()
    assert torch.cuda.is_available(), "bench.py needs a CUDA device"
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inp = dict(workloads.make_inputs(w), linear=w.linear)
    if w.linear:
        inp["beta"] = None  # the linear mode takes no beta (nor copies it end to end)
    d = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in inp.items()}
    B, T, H, dk, dv, C, N = inp["B"], inp["T"], inp["H"], w.dk, w.dv, w.C, inp["N"]
    out = torch.empty((B, T, H, dv), dtype=d["v"].dtype, device=dev)
    Sf = torch.empty((N, H, dv, dk), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        if w.linear:
            gdn.gdn_linear_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["S0"], out, Sf,
                                     C, d["cu_seqlens"], stream=stream)
        else:
            gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["S0"], out,
                              Sf, C, d["cu_seqlens"], stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
        flush.zero_()
    torch.cuda.synchronize()
    gdn.gdn_check_status(stream)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        t_wall0 = time.perf_counter()
        for i in range(args.steps):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
            flush.zero_()
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
    barrier(world)
    gdn.gdn_check_status(stream)
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = sum(per) / len(per)
    ms = max_over_ranks(ms, world, dev)
    alg = algorithmic(dict(inp, C=C))
    tokens = B * T * world
    value = tokens / (ms * 1e-3)
    peaks = load_peaks()
    sec = ms * 1e-3
    achieved_gbs = alg["bytes"] / sec / 1e9
    achieved_tf = alg["flops"] / sec / 1e12
    path = gdn.gdn_select_path(dk, dv, C, d["v"].dtype)
    launches = gdn.gdn_launches_per_call(dk, dv, C, d["v"].dtype)
    scope = "one launch"
    if w.linear and inp["cu_seqlens"] is None and \
            gdn.gdn_linear_split_segments(B, H, T, dk, dv, C, d["v"].dtype) > 1:
        launches = 2  # the segments, then the fold and correction
        scope = "the step's two launches (segments, then fold and correction) against the path's algorithmic bytes"
    elif launches > 1:
        scope = f"the step's {launches} launches against the path's algorithmic bytes"

    # ---- end to end through the public call with pinned host buffers ----
    host_in = {k: (inp[k].pin_memory() if inp[k] is not None else None)
               for k in ("q", "k", "v", "log_alpha", "beta", "S0", "cu_seqlens")}
    out_h = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    Sf_h = torch.empty(Sf.shape, dtype=Sf.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host_in.values() if t is not None)
    d2h = out_h.numel() * out_h.element_size() + Sf_h.numel() * Sf_h.element_size()

    def e2e_step():
        # the public call on pinned host tensors: copies in, computes, copies back,
        # pipelined over token ranges, and synchronises before it returns
        if w.linear:
            return gdn.linear_chunk_fwd(host_in["q"], host_in["k"], host_in["v"],
                                        host_in["log_alpha"], host_in["S0"],
                                        host_in["cu_seqlens"], C=C)
        return gdn.chunk_fwd(host_in["q"], host_in["k"], host_in["v"], host_in["log_alpha"],
                             host_in["beta"], host_in["S0"], host_in["cu_seqlens"], C=C)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    t_e2e = time.perf_counter()
    for _ in range(args.e2e_steps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks((time.perf_counter() - t_e2e) * 1e3 / args.e2e_steps, world, dev)
    gdn.gdn_check_status(stream)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, sample, _ = cpu_oracle_time(inp)
        cpu = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample}

    if rank == 0:
        line = {
            "metric": LINEAR_METRIC if w.linear else METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if path == gdn.GDN_PATH_TCGEN05 else "f32",
            "data": "synthetic",
            "config": {"workload": w.name, "B": B, "H": H, "T": T, "dk": dk, "dv": dv, "C": C,
                       "seqs": N, "qkv_dtype": w.dtype,
                       "path": {1: "recurrence (CUDA cores)", 2: "tcgen05",
                                3: "chunk form, tcgen05 three-pass TF32"}.get(path, "none"),
                       "l2": "flushed between timed steps (512 MiB write)",
                       "parallelism": f"replicas{world}"},
            "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": achieved_gbs / peaks["hbm_gbs"],
                         "traffic": measured_traffic(w.name) if args.T == 0 else None,
                         "peak_source": peaks["source"],
                         "algorithmic_bytes": alg["bytes"], "scope": scope,
                         "tensor_tflops": achieved_tf,
                         "tensor_frac": achieved_tf / peaks["bf16_tflops"]},
            "clocks": clk.summary(),
            "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms,
                    "timing": "host clock around the synchronous public call chunk_fwd on pinned host tensors (copies pipelined over 4 token ranges)"},
            "gpu_launches": launches * args.steps,
            "cpu_baseline": cpu,
            "wall_s_timed_region": t_wall,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
