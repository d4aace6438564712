#!/usr/bin/env python
"""Decode throughput of the MoE channel reader on one GPU (or N replicas).

One step = one decode of every batch size in --batches on each of --layers
distinct prepared Qwen3-30B-A3B-shaped layers (H 2048, E 128, top-8, I 768,
k 756 = the 17.8% read budget, c 80, r 32).  Cycling the layers keeps the
data a step touches (hundreds of MB) far above the 129 MB L2, so no decode
finds its weights in L2.  Every step is one CUDA-graph replay per batch size;
timing uses CUDA events on the replay stream.  The same layers are also run
as one residual-carrying stack per call (the 48-layer stack workload at the
17.8% and 12.8% budgets, batch 1 and 8), reported beside the headline.

Prints ONE JSON line (rank 0).  --impl reference times the fp64 oracle on
the host cores instead (the reference arm: there is no runnable reference
implementation of this method).
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer decode tokens/s at batch 1–16; achieved HBM GB/s vs GB300 peak"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--layers", type=int, default=48)
    ap.add_argument("--batches", default="1,4,8,16")
    ap.add_argument("--input-sets", type=int, default=4)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-stack", action="store_true")
    ap.add_argument("--no-shared", action="store_true")
    ap.add_argument("--no-rho-rank", action="store_true",
                    help="skip the full-screen expected-error ranking (screen_coords 128, "
                         "28.7%% budget)")
    ap.add_argument("--no-large-batch", action="store_true",
                    help="skip the GPT-OSS-120B-shaped layer at batch 1-128 (per-token against "
                         "batch-shared selection)")
    ap.add_argument("--no-235b", action="store_true",
                    help="skip the Qwen3-235B-A22B-shaped layer at the 12.8%% budget")
    ap.add_argument("--no-trit5", action="store_true",
                    help="skip the five-trits-per-byte sketch layout on Qwen3-30B-shaped layers")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu_index), "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(value, world):
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_step, steps, elapsed_ms, world):
    """Whole-job rate of N independent replicas: every rank decodes the same
    fixed work, the job ends when the slowest rank does (max over ranks)."""
    slowest_ms = max_over_ranks(elapsed_ms, world)
    return tokens_per_step * steps * world / (slowest_ms / 1000.0), slowest_ms


# ---------------------------------------------------------------------------
# the oracle on host cores (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------
def oracle_layer_from_bits(wl, G, V, D, sigma):
    from oracle import reader as R

    shape = R.Shape(H=wl.H, E=wl.E, topk=wl.topk, I=wl.I, c=wl.c, r=wl.r)
    return R.Layer(shape, G, V, D, sigma)


def time_oracle(layer, tokens, k, budget_s, min_tokens=1):
    """Decode tokens one by one with the oracle until budget_s has passed.
    Load-time work (U, b, sketches of the experts used) is done first."""
    from oracle import reader as R

    _ = layer.U
    for x, ids, w in tokens:
        for e in ids:
            layer.sketch(int(e))
            layer.b(int(e))
            layer.dnorm(int(e))
    n = 0
    t0 = time.perf_counter()
    for x, ids, w in tokens:
        R.decode_token(layer, x, ids, w, k)
        n += 1
        if n >= min_tokens and time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return n, dt


def cpu_threads():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            try:
                return int(os.environ[var])
            except ValueError:
                pass
    return os.cpu_count() or 1


def sample_tokens(wl, n, seed):
    from calibration_free_sparse_gb300 import synthetic as S

    x = S.activations(seed, n, wl.H)
    ids, w = S.routing(seed, n, wl.E, wl.topk)
    return [(x[i], ids[i], w[i]) for i in range(n)]


def host_layer_bits(wl, seed):
    """Weights of one benchmark layer as host BF16 bit patterns."""
    from calibration_free_sparse_gb300 import synthetic as S

    try:
        import torch

        if torch.cuda.is_available():
            g, v, d = S.weights_device(seed, wl.E, wl.I, wl.H, "cuda")
            out = tuple(S.bf16_tensor_to_bits(t) for t in (g, v, d))
            del g, v, d
            torch.cuda.empty_cache()
            return out
    except ImportError:
        pass
    return S.weights(seed, wl.E, wl.I, wl.H)


def run_reference(args, wl, world, rank):
    if rank != 0:
        return
    from calibration_free_sparse_gb300 import synthetic as S

    seed = 1000
    G, V, D = host_layer_bits(wl, seed)
    layer = oracle_layer_from_bits(wl, G, V, D, S.signs(seed, wl.Hp))
    toks = sample_tokens(wl, args.warmup + args.steps, 77)
    # load-time work and warm-up steps
    time_oracle(layer, toks[: max(1, args.warmup)], wl.k, budget_s=1e9, min_tokens=len(toks))
    n, dt = time_oracle(layer, toks[args.warmup:], wl.k, budget_s=1e9,
                        min_tokens=len(toks) - args.warmup)
    value = n / dt
    cores = cpu_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * dt / max(n, 1), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "H": wl.H, "E": wl.E, "topk": wl.topk, "I": wl.I,
                   "k": wl.k, "c": wl.c, "r": wl.r,
                   "note": "each step decodes one token with the fp64 oracle; the oracle "
                           "is per token, so its cost does not depend on the batch size"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} single-token decodes of one layer"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
PHASE_BYTES = {   # algorithmic parameter arrays each decode kernel reads
    "decode": ("codes", "scales", "dnorm", "G", "V", "Dt", "b", "U"),
}


def kernel_code_digest():
    """sha256[:16] of the decode kernel's code: decode.cu and the headers it
    includes, with comments and whitespace removed (a comment edit keeps a
    recorded capture valid, a code edit does not)."""
    import hashlib
    import re

    h = hashlib.sha256()
    for name in ("decode.cu", "device_util.cuh", "internal.cuh"):
        path = os.path.join(ROOT, "calibration_free_sparse_gb300", "csrc", name)
        with open(path, encoding="utf-8") as f:
            txt = f.read()
        txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
        txt = re.sub(r"//[^\n]*", "", txt)
        h.update(re.sub(r"\s+", "", txt).encode())
    return h.hexdigest()[:16]


def traffic_for(kernel, batch):
    """Per-launch DRAM bytes of `kernel` at `batch` from a committed ncu summary,
    if the summary was taken on the current kernel code."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    ent = rec.get(kernel)
    if not ent or ent.get("code_sha256_16") != kernel_code_digest() or ent.get("batch") != batch:
        return None
    return ent.get("bytes_per_launch")


def layer_sweep(torch, dev, stream, args, wl, k, batches, nl, seed0, modes=("per_token",),
                screen_coords=None, flags=0):
    """Decode time of nl prepared layers of workload wl at each batch (one CUDA
    graph per (mode, batch) cycling the layers, so their weights are not in
    L2), with the sector-accounted bytes of every layer's decode: microseconds
    per decode, layer-tokens/s, read fraction, GB/s and its fraction of the
    measured copy bandwidth."""
    from calibration_free_sparse_gb300 import synthetic as S
    from calibration_free_sparse_gb300.reader import MoeReader

    c = wl.c if screen_coords is None else screen_coords
    readers, keep = [], []
    for l in range(nl):
        g, v, d = S.weights_device(seed0 + l, wl.E, wl.I, wl.H, dev)
        readers.append(MoeReader(wl.H, wl.E, wl.topk, wl.I, g, v, d, S.signs(seed0 + l, wl.Hp),
                                 screen_coords=c, rank=wl.r, max_batch=max(batches), flags=flags))
        keep.append((g, v))
        del d
    torch.cuda.empty_cache()
    peak, _ = measured_peaks()
    info = readers[0].info()
    out = {"workload": wl.name, "H": wl.H, "E": wl.E, "topk": wl.topk, "I": wl.I, "k": k,
           "screen_coords": c, "r": wl.r, "layers": nl, "per_batch": {},
           "resident_sketch_bytes_per_layer": info["resident_bytes"][0] + info["resident_bytes"][1],
           "run_stride": info["run_stride"]}
    for B in batches:
        xs, idw = [], []
        for l in range(nl):
            sd = seed0 + 50_000 + 100 * B + l
            xs.append(torch.from_numpy(S.activations(sd, B, wl.H)).to(dev))
            ids, w = S.routing(sd, B, wl.E, wl.topk)
            idw.append((torch.from_numpy(ids).to(dev), torch.from_numpy(w).to(dev)))
        y = torch.empty((B, wl.H), device=dev)
        row = {}
        for mode in modes:
            def run(mode=mode):
                for l, rd in enumerate(readers):
                    fn = rd.decode_shared if mode == "shared" else rd.decode
                    fn(xs[l], idw[l][0], idw[l][1], k, y)
            sbytes = dbytes = 0
            with torch.cuda.stream(stream):
                for l, rd in enumerate(readers):
                    fn = rd.decode_shared if mode == "shared" else rd.decode
                    fn(xs[l], idw[l][0], idw[l][1], k, y)
                    st = rd.stats()
                    sbytes += 32 * sum(st[a] for a in ("codes", "scales", "dnorm", "G", "V", "Dt",
                                                        "b", "U"))
                    dbytes += 32 * st["dense"]
                    code, bits = rd.status()
                    if code != 0:
                        raise RuntimeError(f"{wl.name} {mode}: device status {code} bits {bits}")
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                run()
            with torch.cuda.stream(stream):
                for _ in range(3):
                    graph.replay()
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            reps = max(3, min(args.steps, 10))
            with torch.cuda.stream(stream):
                ev0.record(stream)
                for _ in range(reps):
                    graph.replay()
                ev1.record(stream)
            torch.cuda.synchronize()
            us = 1000.0 * ev0.elapsed_time(ev1) / (reps * nl)
            gbs = (sbytes / nl) / (us * 1e-6) / 1e9
            row[mode] = {"us_per_decode": us, "tokens_per_s": B / (us * 1e-6),
                         "sector_bytes_per_decode": sbytes / nl, "read_fraction": sbytes / dbytes,
                         "hbm_gbs": gbs, "frac_of_measured_peak": gbs / peak}
        if "shared" in row and "per_token" in row:
            row["shared"]["vs_per_token"] = row["per_token"]["us_per_decode"] / row["shared"]["us_per_decode"]
        out["per_batch"][str(B)] = row if len(modes) > 1 else row[modes[0]]
    for rd in readers:
        rd.close()
    del keep
    torch.cuda.empty_cache()
    return out


def run_ours(args, wl, world, rank, local):
    import torch

    from calibration_free_sparse_gb300 import synthetic as S
    from calibration_free_sparse_gb300.reader import PHASES, MoeReader

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    batches = [int(b) for b in args.batches.split(",")]
    Bmax = max(batches)
    L = args.layers
    nsets = max(1, args.input_sets)

    # -- prepared layers (weights drawn on the device, one seed per layer and rank)
    readers, keep = [], []
    prep_s = []
    for l in range(L):
        seed = 1000 + l + 7919 * rank
        g, v, d = S.weights_device(seed, wl.E, wl.I, wl.H, dev)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        rd = MoeReader(wl.H, wl.E, wl.topk, wl.I, g, v, d, S.signs(seed, wl.Hp),
                       screen_coords=wl.c, rank=wl.r, max_batch=Bmax)   # synchronizes its stream
        prep_s.append(time.perf_counter() - t0)
        del d
        readers.append(rd)
        keep.append((g, v))
    torch.cuda.empty_cache()

    # -- inputs: nsets distinct sets per (batch, layer)
    inputs = {}
    for si in range(nsets):
        for B in batches:
            for l in range(L):
                sd = 10_000 * (si + 1) + 100 * B + l + 7919 * rank
                x = S.activations(sd, B, wl.H)
                ids, w = S.routing(sd, B, wl.E, wl.topk)
                inputs[(si, B, l)] = (torch.from_numpy(x).to(dev), torch.from_numpy(ids).to(dev),
                                      torch.from_numpy(w).to(dev), torch.empty((B, wl.H), device=dev),
                                      (x, ids, w))

    # -- algorithmic bytes per decode (library read accounting, per phase)
    stream = torch.cuda.Stream(device=dev)
    phase_bytes = {B: {p: 0 for p in PHASE_BYTES} for B in batches}
    sector_bytes = {B: 0 for B in batches}
    dense_bytes = {B: 0 for B in batches}
    with torch.cuda.stream(stream):
        for B in batches:
            for l, rd in enumerate(readers):
                x, ids, w, y, _ = inputs[(0, B, l)]
                rd.decode(x, ids, w, wl.k, y)
                st = rd.stats()
                for p, arrs in PHASE_BYTES.items():
                    phase_bytes[B][p] += 32 * sum(st[a] for a in arrs)
                sector_bytes[B] += 32 * sum(st[a] for a in ("codes", "scales", "dnorm", "G", "V",
                                                             "Dt", "b", "U"))
                dense_bytes[B] += 32 * st["dense"]
                code, bits = rd.status()
                if code != 0:
                    raise RuntimeError(f"device status {code} bits {bits}")

    # -- CUDA graphs: one per (input set, batch), each decoding every layer
    def capture(si, B):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for l, rd in enumerate(readers):
                x, ids, w, y, _ = inputs[(si, B, l)]
                rd.decode(x, ids, w, wl.k, y)
        return graph

    torch.cuda.synchronize()
    graphs = {(si, B): capture(si, B) for si in range(nsets) for B in batches}
    launches_per_decode = 1
    launches_per_step = launches_per_decode * L * len(batches)

    def step(i, events=None):
        si = i % nsets
        for bi, B in enumerate(batches):
            if events is not None:
                events[bi][0].record(stream)
            graphs[(si, B)].replay()
            if events is not None:
                events[bi][1].record(stream)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    torch.cuda.synchronize()

    # -- timed region
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit() else local
    clocks = ClockSampler(gpu_index)
    per_b_events = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                     for _ in batches] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.25)
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for i in range(args.steps):
            step(i, per_b_events[i])
        t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    time.sleep(0.15)
    clk = clocks.stop()
    elapsed_ms = t_start.elapsed_time(t_end)
    per_b_ms = {B: sum(per_b_events[i][bi][0].elapsed_time(per_b_events[i][bi][1])
                       for i in range(args.steps)) for bi, B in enumerate(batches)}
    tokens_per_step = L * sum(batches)
    value, elapsed_ms = job_throughput(tokens_per_step, args.steps, elapsed_ms, world)

    # -- per-phase device time (profiling events inside fresh graphs of set 0)
    for rd in readers:
        rd.set_profiling(True)
    prof_graphs = {B: capture(0, B) for B in batches}
    prof_steps = min(args.steps, 50)
    phase_ms = {B: {p: 0.0 for p in PHASES} for B in batches}
    for _ in range(prof_steps):
        with torch.cuda.stream(stream):
            for B in batches:
                prof_graphs[B].replay()
        for rd in readers:
            rows = rd.read_profile()          # slot bi = the decode captured for batches[bi]
            for bi, B in enumerate(batches):
                for p in PHASES:
                    phase_ms[B][p] += rows[bi][p]
    for rd in readers:
        rd.set_profiling(False)

    peak, peak_kind = measured_peaks()
    per_batch = {}
    for B in batches:
        ms_decode = per_b_ms[B] / (args.steps * L)
        gbs = (sector_bytes[B] / L) / (ms_decode / 1000.0) / 1e9
        per_batch[str(B)] = {
            "tokens_per_s": B / (ms_decode / 1000.0),
            "us_per_decode": 1000.0 * ms_decode,
            "sector_bytes_per_decode": sector_bytes[B] / L,
            "read_fraction": sector_bytes[B] / dense_bytes[B],
            "hbm_gbs": gbs,
            "frac_of_measured_peak": gbs / peak,
            "frac_of_nominal_8tbs": gbs / NOMINAL_HBM_GBS,
            "phase_us_per_decode": {p: 1000.0 * phase_ms[B][p] / (prof_steps * L) for p in PHASES},
        }
    # the decode is one persistent kernel, the only one; its roofline is given for
    # the largest batch of the sweep (per launch: bytes and time averaged over layers)
    Bd = max(batches)
    dom_bytes = phase_bytes[Bd]["decode"] / L
    dom_ms = phase_ms[Bd]["decode"] / (prof_steps * L)
    achieved = dom_bytes / (dom_ms / 1000.0) / 1e9 if dom_ms > 0 else 0.0
    traffic = traffic_for("decode_kernel", Bd)
    roofline = {"bound": "hbm", "kernel": "decode_kernel", "launch": f"batch {Bd}",
                "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": traffic, "algorithmic_bytes_per_launch": dom_bytes,
                "launch_us": 1000.0 * dom_ms, "peak_kind": f"{peak_kind} copy bandwidth",
                "share_of_step_time": 1.0}

    # -- batch-shared selection (one kept set per batch) on the same layers and
    # inputs: informational, the headline keeps per-token selection
    shared = None
    if not args.no_shared:
        shared = {"per_batch": {}}
        for B in batches:
            def run_shared(B=B):
                for l, rd in enumerate(readers):
                    x, ids, w, y, _ = inputs[(0, B, l)]
                    rd.decode_shared(x, ids, w, wl.k, y)
            with torch.cuda.stream(stream):
                run_shared()
            rd0 = readers[0]
            st = rd0.stats()
            sb = 32 * sum(st[a] for a in ("codes", "scales", "dnorm", "G", "V", "Dt", "b", "U"))
            for rd in readers:
                code, bits = rd.status()
                if code != 0:
                    raise RuntimeError(f"shared: device status {code} bits {bits}")
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                run_shared()
            with torch.cuda.stream(stream):
                for _ in range(max(3, args.warmup)):
                    graph.replay()
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                ev0.record(stream)
                for _ in range(args.steps):
                    graph.replay()
                ev1.record(stream)
            torch.cuda.synchronize()
            us = 1000.0 * ev0.elapsed_time(ev1) / (args.steps * L)
            shared["per_batch"][str(B)] = {
                "us_per_decode": us, "tokens_per_s": B / (us / 1e6),
                "sector_bytes_per_decode_layer0": sb, "read_fraction_layer0": sb / (32 * st["dense"]),
                "vs_per_token": per_batch[str(B)]["us_per_decode"] / us}
        shared["note"] = ("moe_reader_decode_shared on the same %d layers and inputs, one CUDA "
                          "graph per batch: one kept set per batch of k n_e / topk channels" % L)

    # -- the same layers as one stack per call (residual carried on the device):
    # informational, the headline above decodes the layers independently
    stack = None
    if not args.no_stack:
        from calibration_free_sparse_gb300.reader import decode_stack

        stack = {"layers": L, "per_budget": {}}
        k_low = S.QWEN3_30B_LOW.k if wl.name == S.QWEN3_30B.name else None
        budgets = [("17.8%", wl.k)] + ([("12.8%", k_low)] if k_low is not None else [])
        stack_batches = [B for B in batches if B in (1, 8)] or batches
        for (bname, kk), B in [(bk, B) for bk in budgets for B in stack_batches]:
            h_in = inputs[(0, B, 0)][0]
            ids = torch.stack([inputs[(0, B, l)][1] for l in range(L)]).contiguous()
            w = torch.stack([inputs[(0, B, l)][2] for l in range(L)]).contiguous()
            h_out = torch.empty_like(h_in)
            with torch.cuda.stream(stream):
                decode_stack(readers, h_in, ids, w, kk, h_out)
            for rd in readers:
                code, bits = rd.status()
                if code != 0:
                    raise RuntimeError(f"stack: device status {code} bits {bits}")
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                decode_stack(readers, h_in, ids, w, kk, h_out)
            with torch.cuda.stream(stream):
                for _ in range(max(3, args.warmup)):
                    graph.replay()
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                ev0.record(stream)
                for _ in range(args.steps):
                    graph.replay()
                ev1.record(stream)
            torch.cuda.synchronize()
            us_layer = 1000.0 * ev0.elapsed_time(ev1) / (args.steps * L)
            row = {"k": kk, "us_per_layer": us_layer, "tokens_per_s": B / (us_layer / 1e6),
                   "us_per_stack_step": us_layer * L}
            if kk == wl.k:
                row["vs_independent_decodes"] = per_batch[str(B)]["us_per_decode"] / us_layer
            stack["per_budget"].setdefault(bname, {})[str(B)] = row
        stack["note"] = ("moe_reader_decode_stack over the %d prepared layers, one call per "
                         "step captured in a CUDA graph: an input-scale kernel plus one decode "
                         "grid per layer, residual and next input carried on the device; "
                         "vs_independent_decodes compares with the headline's unchained "
                         "per-layer decodes, which carry no residual" % L)

    # -- the other configurations of the workload family, each on its own
    # prepared layers (informational keys; the headline is the Qwen3-30B layer)
    large = q235 = rho = None
    if not args.no_235b:
        wl2 = S.QWEN3_235B
        q235 = layer_sweep(torch, dev, stream, args, wl2, wl2.k, (1, 4, 8, 16), 6,
                           2000 + 7919 * rank)
        q235["budget"] = 0.128
    if not args.no_large_batch:
        wl3 = S.GPT_OSS_120B
        large = layer_sweep(torch, dev, stream, args, wl3, wl3.k, (1, 4, 8, 16, 32, 64, 128), 6,
                            300 + 7919 * rank, modes=("per_token", "shared"))
        large["budget"] = 0.178
    trit5 = None
    if not args.no_trit5:
        from calibration_free_sparse_gb300.reader import FLAG_TRIT5

        trit5 = layer_sweep(torch, dev, stream, args, wl, wl.k, batches, 12, 900 + 7919 * rank,
                            flags=FLAG_TRIT5)
        trit5["budget"] = 0.178
        two = readers[0].info()
        trit5["two_bit_resident_sketch_bytes_per_layer"] = two["resident_bytes"][0] + two["resident_bytes"][1]
        for B in batches:
            row = trit5["per_batch"][str(B)]
            row["vs_two_bit_headline"] = per_batch[str(B)]["us_per_decode"] / row["us_per_decode"]
            row["two_bit_read_fraction"] = per_batch[str(B)]["read_fraction"]
        trit5["note"] = ("MOE_READER_FLAG_TRIT5 on 12 Qwen3-30B-shaped layers: the same decode with "
                         "the sketch stored five trits per byte; vs_two_bit_headline > 1 is faster")
    if not args.no_rho_rank:
        from calibration_free_sparse_gb300.reader import FLAG_RHO_RANK

        rho = layer_sweep(torch, dev, stream, args, wl, S.budget_to_k(0.287, wl.N), batches, 4,
                          700 + 7919 * rank, screen_coords=128, flags=FLAG_RHO_RANK)
        rho["budget"] = 0.287

    # -- end to end through the host-buffer C ABI (pinned host memory)
    e2e = None
    if not args.no_e2e:
        host = {}
        for B in batches:
            for l in range(L):
                x, ids, w = inputs[(0, B, l)][4]
                hx = torch.from_numpy(x).pin_memory()
                hi = torch.from_numpy(ids).pin_memory()
                hw = torch.from_numpy(w).pin_memory()
                hy = torch.empty((B, wl.H), dtype=torch.float32).pin_memory()
                host[(B, l)] = (hx.numpy(), hi.numpy(), hw.numpy(), hy.numpy())
        e2e_steps = max(3, min(args.steps, 20))
        h2d = sum(B * wl.H * 4 + B * wl.topk * 8 for B in batches) * L
        d2h = sum(B * wl.H * 4 + 4 for B in batches) * L

        def host_step():
            for B in batches:
                for l, rd in enumerate(readers):
                    hx, hi, hw, hy = host[(B, l)]
                    rd.decode_host(hx, hi, hw, wl.k, hy, stream=stream)

        host_step()
        torch.cuda.synchronize()
        barrier(world)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            host_step()
        ev1.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        wall = max_over_ranks(wall, world)
        e2e = {"value": tokens_per_step * e2e_steps * world / wall, "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": e2e_steps,
               "note": "moe_reader_decode_host per layer and batch: pinned H2D of x/ids/w, "
                       "decode, D2H of y and the status word, stream synchronize"}

    # -- the oracle on host cores (rank 0, N = 1 only)
    cpu = None
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        G = S.bf16_tensor_to_bits(keep[0][0])
        V = S.bf16_tensor_to_bits(keep[0][1])
        g, v, d = S.weights_device(1000, wl.E, wl.I, wl.H, dev)
        D = S.bf16_tensor_to_bits(d)
        del g, v, d
        layer = oracle_layer_from_bits(wl, G, V, D, S.signs(1000, wl.Hp))
        toks = []
        for B in batches:
            x, ids, w = inputs[(0, B, 0)][4]
            toks += [(x[t], ids[t], w[t]) for t in range(B)]
        # the pool is cycled so that the sample lasts the whole time budget
        n, dt = time_oracle(layer, toks * 64, wl.k, budget_s=args.cpu_seconds)
        cpu = {"value": n / dt, "unit": "tokens/s", "cores": cpu_threads(), "kind": "oracle",
               "sample": f"{n} tokens of layer 0 from the benchmark batches, decoded one at a "
                         f"time by the fp64 oracle in {dt:.1f} s (load-time work excluded)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {
                "workload": wl.name, "H": wl.H, "E": wl.E, "topk": wl.topk, "I": wl.I,
                "k": wl.k, "read_budget": 0.178, "screen_coords": wl.c, "rank": wl.r,
                "batches": batches, "layers_per_step": L, "input_sets": nsets,
                "weights": "bf16 experts + 2-bit ternary sketch (fp16 scales)",
                "l2": "inputs larger than L2: each step decodes on %d distinct prepared "
                      "layers (%.0f MB of sector-accounted reads per step vs 129 MB L2)"
                      % (L, sum(sector_bytes.values()) / 1e6),
                "parallelism": f"replicas x{world}",
                "tokens": "layer-tokens: one token through one MoE layer",
            },
            "per_batch": per_batch,
            "roofline": roofline,
            "stack": stack,
            "shared": shared,
            "qwen3_235b": q235,
            "trit5": trit5,
            "large_batch": large,
            "rho_rank": rho,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "prepare_ms_per_layer": 1000.0 * statistics.median(prep_s),
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    for rd in readers:
        rd.close()


def main():
    args = parse_args()
    world, rank, local = dist_setup()
    from calibration_free_sparse_gb300 import synthetic as S

    wl = S.QWEN3_30B
    if args.impl == "reference":
        run_reference(args, wl, world, rank)
    else:
        run_ours(args, wl, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
