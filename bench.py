#!/usr/bin/env python3
"""Benchmark: gate-first sparse FFN decode throughput on one GB300 (or N replicas).

Workload (one "step"): the decode stream of the standard-gate layer of Figure 2
of "Model Casting and Low-Parameter Gating" -- D=2560, H=7168, bf16 weights,
ReLU gate shifted for 90 % sparsity, B=1 -- 4096 tokens, token t through layer
set t mod 8 (8 independent layer weight sets, 881 MB, far above the 129 MB L2,
so no call finds its weights in L2).  Each token is one sffn_forward call; the
4096 calls of a step are captured once in a CUDA graph and replayed.

Printed (rank 0, one JSON line): tokens/s of the whole job (value), us per
call, achieved HBM GB/s on the bytes the method touches (the gate matrix plus
the live rows of W3 and W2^T, plus x and y) as a fraction of the measured copy
peak and of the nominal 8 TB/s, the same figures for the dense bf16 FFN
(cuBLAS through torch), and for the variants: the low-rank gate layer
(D=2560, H'=9787, r=400, 32 rotated sets) alone and in the full form (tiled
identity G, RMSNorm, double activation), the smooth SiLU gate with a live
threshold, weight-only int8 and int4 weights, batches of 2 tokens (union gathers) and
of 4 / 16 / 64 tokens on the tensor cores for both gates; an end-to-end figure
with host buffers, SM clocks sampled during the timed region, and the fp64 CPU
oracle timed on a bounded sample of the same workload.

--sweep runs the D=4096 sparsity x batch sweep instead (standard gate H=14336
and low-rank gate H'=19649, r=640; s in {0.5, 0.75, 0.9, 0.95}; B in {1, 8,
32, 128}; each point next to the dense bf16 FFN), one JSON line per point.

--impl reference times the reference arm: the fp64 CPU oracle, as it stands,
on the host cores (rank 0 only), on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "std-bf16-D2560-H7168-B1"
LOPA_WORKLOAD = "lopa-bf16-D2560-H9787-r400-B1"
METRIC = "sparse-FFN tokens/s & µs/call at B=1 (HBM GB/s vs 8 TB/s) vs dense bf16 FFN"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ("activation_sparse_gated_gb300/csrc/ffn_b1_bf16.cu",
                  "activation_sparse_gated_gb300/csrc/common.cuh")
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "ffn_b1_bf16_std_D2560_H7168.md")


def kernel_hash() -> str:
    """Hash of the dominant kernel's source, to tie committed ncu counters to it."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def ncu_traffic_per_launch():
    """DRAM bytes per launch from the committed ncu summary, if taken on this kernel source."""
    try:
        text = open(PROFILE_SUMMARY).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel source hash:\s*`?([0-9a-f]{16})", text)
    m_bytes = re.search(r"dram bytes per launch:\s*([0-9.]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != kernel_hash():
        return None
    return float(m_bytes.group(1))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None
        self.fh = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.fh:
            self.fh.close()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                f = [c.strip() for c in line.split(",")]
                if len(f) >= 9 and f[1].replace(".", "").isdigit():
                    rows.append(f)
        finally:
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        smax = max(float(r[2]) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        loaded = [v for v in sm if v > 0.5 * smax] or sm
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(power) if power else None}


# --------------------------------------------------------------------------- CPU oracle timing
def time_oracle(layers, x, budget_s: float, max_tokens: int):
    """Oracle over a bounded sample: tokens in order, token t through set t mod len(layers)."""
    import oracle
    from activation_sparse_gated_gb300 import synthetic as syn
    views = [{k: syn.oracle_view(t) for k, t in lw.tensors().items()} for lw in layers]
    lw0 = layers[0]
    n, t0 = 0, time.perf_counter()
    while n < max_tokens:
        v = views[n % len(views)]
        oracle.ffn_dense(lw0.D, lw0.H, lw0.r, oracle.RELU, oracle.BF16, v["W1"], v["U"], v["V"],
                         v["W3"], v["W2"], syn.oracle_view(x[n:n + 1]))
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    return n, time.perf_counter() - t0, oracle.num_threads()


def oracle_one_thread(budget_s: float):
    """The same oracle sample on one OpenMP thread (a child process with OMP_NUM_THREADS=1)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", RANK="0", WORLD_SIZE="1")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-one-thread", str(budget_s)],
                           env=env, capture_output=True, text=True, timeout=300)
        d = json.loads(r.stdout.strip().splitlines()[-1])
    except (subprocess.SubprocessError, ValueError, IndexError, OSError):
        return None
    return {"value": d["tokens"] / d["seconds"], "unit": "tokens/s", "cores": d["cores"],
            "sample": f"first {d['tokens']} tokens, {d['seconds']:.1f} s"}


def run_reference(args):
    """The reference arm: the fp64 oracle on the host cores, rank 0 only."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    import oracle
    from activation_sparse_gated_gb300 import synthetic as syn
    oracle.build()
    sets, per_step = 2, 8
    layers = syn.workload_layers(WORKLOAD, sets=sets)
    x = syn.workload_tokens(WORKLOAD, per_step * (args.steps + args.warmup))
    for w in range(args.warmup):
        time_oracle(layers, x[w * per_step:(w + 1) * per_step], 1e9, per_step)
    t0, done, cores = time.perf_counter(), 0, 1
    for k in range(args.steps):
        s = (args.warmup + k) * per_step
        n, _, cores = time_oracle(layers, x[s:s + per_step], 1e9, per_step)
        done += n
    dt = time.perf_counter() - t0
    value = done / dt
    sample = (f"{per_step} tokens per step of the {WORKLOAD} decode stream, token t through "
              f"weight set t mod {sets}, fp64 dense oracle (OpenMP)")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "D": 2560, "H": 7168, "B": 1, "tokens_per_step": per_step,
                   "weight_sets": sets},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# --------------------------------------------------------------------------- GPU arm
def build_ffns(layers, dev, flags=0, act="relu", thr=0.0, dtype=None):
    import activation_sparse_gated_gb300 as sffn
    ffns = []
    for lw in layers:
        f = sffn.SparseFFN(lw.D, lw.H, lw.r, act, dtype or lw.dtype, flags=flags)
        if thr:
            f.set_live_threshold(thr)
        w = {k: (None if t is None else t.to(dev)) for k, t in lw.tensors().items()}
        f.set_weights(w["W1"] if lw.r == 0 else w["U"], w["V"], w["W3"], w["W2"])
        del w
        ffns.append(f)
    return ffns


def live_counts(ffns, x, stream):
    """Live units per call for the step's token order (untimed, one synchronising pass)."""
    import torch
    import activation_sparse_gated_gb300 as sffn
    y = torch.empty_like(x[:1])
    counts = []
    with torch.cuda.stream(stream):
        for t in range(x.shape[0]):
            f = ffns[t % len(ffns)]
            sffn.sffn_forward(f.h, x[t], y, 1, stream)
            counts.append(f.active_counts(1)[0])
    return counts


def capture_step(ffns, x, y, stream):
    import torch
    import activation_sparse_gated_gb300 as sffn
    n = x.shape[0]
    with torch.cuda.stream(stream):          # eager warm-up of every handle
        for t in range(len(ffns)):
            sffn.sffn_forward(ffns[t].h, x[t], y[t], 1, stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for t in range(n):
            sffn.sffn_forward(ffns[t % len(ffns)].h, x[t], y[t], 1, stream)
    return g


def replica_totals(t_local, units_per_rank, world, dist=None, device=None):
    """Whole-job figures of N weakly scaled replicas (one rank per GPU, no data
    exchange): the timed region ends when the slowest rank ends, so the job's
    time is the maximum over ranks, and its throughput is the units all ranks
    processed divided by that time.  Returns (seconds, units per second)."""
    t = float(t_local)
    if dist is not None and world > 1:
        import torch
        tt = torch.tensor([t], device=device, dtype=torch.float64)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        t = float(tt.item())
    return t, world * units_per_rank / t


def time_graph(g, stream, steps, warmup, dist=None):
    import torch
    for _ in range(warmup):
        g.replay()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    return e0.elapsed_time(e1) / 1e3


def dense_graphs(layers_dev, x, y, stream):
    """Dense bf16 FFN via cuBLAS (torch), same token/set order; the 3-GEMV and concatenated forms."""
    import torch
    import torch.nn.functional as F
    n = x.shape[0]
    H = layers_dev[0]["W1"].shape[0]
    graphs = {}
    for form in ("three", "concat"):
        def body():
            for t in range(n):
                L = layers_dev[t % len(layers_dev)]
                xt = x[t:t + 1]
                if form == "three":
                    h = F.relu(F.linear(xt, L["W1"])) * F.linear(xt, L["W3"])
                else:
                    zu = F.linear(xt, L["W13"])
                    h = F.relu(zu[:, :H]) * zu[:, H:]
                y[t:t + 1] = F.linear(h, L["W2"])
        with torch.cuda.stream(stream):
            body()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            body()
        graphs[form] = g
    return graphs


def batched_extras(ffns, layers, x, stream, args, peak):
    """Batched decode of the same layer sets: B tokens per call, token group t through set t mod 8."""
    import torch
    import torch.nn.functional as F
    import activation_sparse_gated_gb300 as sffn
    D, H = layers[0].D, layers[0].H
    dev = x.device
    n_sets = len(ffns)
    ld = [{"W1": lw.W1.to(dev), "W3": lw.W3.to(dev), "W2": lw.W2.to(dev)} for lw in layers]
    out = {}
    for B in (2, 4, 8, 16, 64):
        calls = x.shape[0] // B
        y = torch.empty_like(x)
        # union of the tokens' live sets per call (untimed)
        unions = []
        with torch.cuda.stream(stream):
            for t in range(min(calls, 64)):
                f = ffns[t % n_sets]
                sffn.sffn_forward(f.h, x[t * B:(t + 1) * B], y[t * B:(t + 1) * B], B, stream)
                unions.append(int(f.active_mask(B).any(axis=0).sum()))
        stream.synchronize()
        mean_union = sum(unions) / len(unions)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for t in range(calls):
                sffn.sffn_forward(ffns[t % n_sets].h, x[t * B:(t + 1) * B], y[t * B:(t + 1) * B], B, stream)
        tt = time_graph(g, stream, args.steps, args.warmup)
        us = 1e6 * tt / (args.steps * calls)
        # B = 2 gathers the union of the live sets (gate on the tensor cores, union rows of W3 and
        # W2^T on the CUDA cores): W1 + the union rows + x, y.  Larger batches of this shape stream
        # every unit slice of W1, W3 and W2 plus x, y and h (bf16, written once, read once): here
        # the union-skip kernels would save less than 128 MB a call, below what pays on this GPU (they
        # run when forced through SFFN_TCG_MAX_BATCH: W1, the union rows of W3 and W2^T, x, y, the
        # union's h and the union list).  union_gather_bytes is what a row-gathering design reads.
        union_path = 2 <= B <= int(os.environ.get("SFFN_TCU_MAX_BATCH", "2"))
        skip_path = not union_path and 3 <= B <= int(os.environ.get("SFFN_TCG_MAX_BATCH", "0"))
        tc_path = B >= int(os.environ.get("SFFN_TC_MIN_BATCH", "2")) and not union_path and not skip_path
        union_bytes = 2 * H * D + 2 * 2 * mean_union * D + 2 * 2 * B * D
        skip_bytes = union_bytes + 2 * 2 * B * mean_union + 2 * 4 * mean_union
        bytes_call = ((3 * 2 * H * D + 2 * 2 * B * D + 2 * 2 * B * H) if tc_path else
                      skip_bytes if skip_path else union_bytes)
        yd = torch.empty_like(x)

        def body():
            for t in range(calls):
                L = ld[t % n_sets]
                xt = x[t * B:(t + 1) * B]
                yd[t * B:(t + 1) * B] = F.linear(F.relu(F.linear(xt, L["W1"])) * F.linear(xt, L["W3"]), L["W2"])
        with torch.cuda.stream(stream):
            body()
        stream.synchronize()
        gd = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gd, stream=stream):
            body()
        td = time_graph(gd, stream, args.steps, args.warmup)
        usd = 1e6 * td / (args.steps * calls)
        path = ("tensor cores: gate-up + down kernels" if tc_path else
                "tensor cores, union skip: gate kernel (W1, then the union's W3 rows) + down kernel"
                if skip_path else
                "union gathers: gate on the tensor cores, union rows on the CUDA cores" if union_path else
                "CUDA cores, union gathers")
        out[f"B{B}"] = {"path": path,
                        "us_per_call": us, "tokens_per_s": B * 1e6 / us, "mean_union_units": mean_union,
                        "union_fraction": mean_union / H, "bytes_per_call": bytes_call,
                        "union_gather_bytes": union_bytes, "gbs": bytes_call / (us * 1e3),
                        "frac_of_measured": bytes_call / (us * 1e3) / peak,
                        "dense_bf16_us_per_call": usd, "speedup_vs_dense_bf16": usd / us,
                        "gpu_launches_per_call": 2 if tc_path else 2 * ((B + 7) // 8)}
        del g, gd
    return out


def union_skip_extras(stream, args, peak, dev, gate, name, s, B, n_sets):
    """The union-skip kernels where they pay, against the streaming kernels on the same weights (the
    live-fraction hint picks the path): `gate` layer of workload `name` with its bias rewritten for
    sparsity s, B tokens per call over n_sets rotated weight sets."""
    import torch
    import activation_sparse_gated_gb300 as sffn
    from activation_sparse_gated_gb300 import synthetic as syn
    w = syn.WORKLOADS[name]
    D = w["D"]
    layers = syn.workload_layers(name, sets=n_sets, gate=gate, s=s)
    H, r = layers[0].H, layers[0].r
    x = syn.workload_tokens(name).to(dev)
    x = x[:min(x.shape[0], 1024)]
    calls = x.shape[0] // B
    out = {"workload": f"{name} {gate} gate, s = {s}, B = {B}, {n_sets} rotated weight sets"}
    for path, rho in (("union_skip", 1.0 - s), ("streaming", -1.0)):
        ffns = build_ffns(layers, dev)
        for f in ffns:
            f.set_live_fraction_hint(rho)
        y = torch.empty_like(x)
        unions = []
        with torch.cuda.stream(stream):
            for t in range(min(calls, 32)):
                f = ffns[t % n_sets]
                sffn.sffn_forward(f.h, x[t * B:(t + 1) * B], y[t * B:(t + 1) * B], B, stream)
                unions.append(int(f.active_mask(B).any(axis=0).sum()))
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for t in range(calls):
                sffn.sffn_forward(ffns[t % n_sets].h, x[t * B:(t + 1) * B], y[t * B:(t + 1) * B], B, stream)
        us = 1e6 * time_graph(g, stream, args.steps, args.warmup) / (args.steps * calls)
        u = sum(unions) / len(unions)
        gate_bytes = 2 * H * D if r == 0 else 2 * r * (D + H) + 2 * 2 * B * r  # W1, or V, U and the t pair
        if path == "union_skip":
            nbytes = gate_bytes + 2 * 2 * u * D + 2 * 2 * B * D + 2 * 2 * B * u + 2 * 4 * u
        else:
            nbytes = gate_bytes + 2 * 2 * H * D + 2 * 2 * B * D + 2 * 2 * B * H
        out[path] = {"us_per_call": us, "tokens_per_s": B * 1e6 / us, "mean_union_units": u,
                     "union_fraction": u / H, "bytes_per_call": nbytes, "gbs": nbytes / (us * 1e3),
                     "frac_of_measured": nbytes / (us * 1e3) / peak,
                     "gpu_launches_per_call": 2 if r == 0 else 3}
        del g, ffns
    out["speedup_union_skip_vs_streaming"] = out["streaming"]["us_per_call"] / out["union_skip"]["us_per_call"]
    return out


def lopa_batched_extras(ffns, x, stream, args, peak, D, Hp, r):
    """Batched decode of the low-rank layer sets on the tensor cores: t as a bf16 pair, the gate
    U t and the up projection in one gate-up kernel, the down kernel; B tokens per call."""
    import torch
    import activation_sparse_gated_gb300 as sffn
    out = {}
    n_sets = len(ffns)
    for B in (4, 16, 64):
        calls = x.shape[0] // B
        y = torch.empty_like(x)
        unions = []
        with torch.cuda.stream(stream):
            for t in range(min(calls, 64)):
                f = ffns[t % n_sets]
                sffn.sffn_forward(f.h, x[t * B:(t + 1) * B], y[t * B:(t + 1) * B], B, stream)
                unions.append(int(f.active_mask(B).any(axis=0).sum()))
        stream.synchronize()
        mean_union = sum(unions) / len(unions)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for t in range(calls):
                sffn.sffn_forward(ffns[t % n_sets].h, x[t * B:(t + 1) * B], y[t * B:(t + 1) * B], B, stream)
        us = 1e6 * time_graph(g, stream, args.steps, args.warmup) / (args.steps * calls)
        del g
        # streamed: U, V and every slice of W3 and W2^T, plus x, y, the t pair and h
        streamed = 2 * r * (D + Hp) + 2 * 2 * Hp * D + 2 * 2 * B * D + 2 * 2 * B * r + 2 * 2 * B * Hp
        union_bytes = 2 * r * (D + Hp) + 2 * 2 * mean_union * D + 2 * 2 * B * D
        out[f"B{B}"] = {"path": "tensor cores: t pair, gate-up (U t and W3 x) + down kernels",
                        "us_per_call": us, "tokens_per_s": B * 1e6 / us, "mean_union_units": mean_union,
                        "union_fraction": mean_union / Hp, "bytes_per_call": streamed,
                        "union_gather_bytes": union_bytes, "gbs": streamed / (us * 1e3),
                        "frac_of_measured": streamed / (us * 1e3) / peak, "gpu_launches_per_call": 3}
    return out


def run_gpu(args):
    import torch
    import activation_sparse_gated_gb300 as sffn
    from activation_sparse_gated_gb300 import build as libbuild
    from activation_sparse_gated_gb300 import synthetic as syn
    from oracle import flops

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    torch.cuda.set_device(local)
    dev = torch.device(f"cuda:{local}")
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    libbuild.build()
    sffn.load()

    info = syn.WORKLOADS[WORKLOAD]
    D, H, n_tok, n_sets = info["D"], info["H"], info["tokens"], info["sets"]
    layers = syn.workload_layers(WORKLOAD)
    ffns = build_ffns(layers, dev)
    x_host = syn.workload_tokens(WORKLOAD)
    x = x_host.to(dev)
    y = torch.empty_like(x)
    stream = torch.cuda.Stream(device=dev)

    counts = live_counts(ffns, x, stream)
    mean_live = sum(counts) / len(counts)
    elt = 2
    # algorithmic bytes of one call: W1 + the live rows of W3 and W2^T + x + y
    bytes_step = float(sum(elt * H * D + 2 * elt * k * D + 2 * elt * D for k in counts))

    g = capture_step(ffns, x, y, stream)
    peak, peak_kind = measured_peaks()
    with ClockSampler(local) as clk:
        t = time_graph(g, stream, args.steps, args.warmup, dist)
    clocks = clk.summary()
    t, value = replica_totals(t, args.steps * n_tok, world, dist, dev)
    us_call = 1e6 * t / (args.steps * n_tok)
    achieved = bytes_step * args.steps / (t * 1e9)   # per GPU

    # eager launches (no graph): the same step through the C ABI from Python
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for tk in range(n_tok):
            sffn.sffn_forward(ffns[tk % n_sets].h, x[tk], y[tk], 1, stream)
        e1.record(stream)
    torch.cuda.synchronize()
    us_call_eager = 1e3 * e0.elapsed_time(e1) / n_tok

    # end to end: pinned host tokens in, outputs back to pinned host memory, every step
    xh = x_host.pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            x.copy_(xh, non_blocking=True)
            g.replay()
            yh.copy_(y, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    t_e2e, v_e2e = replica_totals(e0.elapsed_time(e1) / 1e3, args.steps * n_tok, world, dist, dev)
    e2e = {"value": v_e2e, "unit": "tokens/s",
           "h2d_bytes_per_step": xh.numel() * xh.element_size(),
           "d2h_bytes_per_step": yh.numel() * yh.element_size()}

    extras = {}
    if not args.no_extras:
        ld = []
        for lw in layers:
            W1, W3, W2 = lw.W1.to(dev), lw.W3.to(dev), lw.W2.to(dev)
            ld.append({"W1": W1, "W3": W3, "W2": W2, "W13": torch.cat([W1, W3], 0)})
        yd = torch.empty_like(x)
        dg = dense_graphs(ld, x, yd, stream)
        dense_t = {k: time_graph(gr, stream, args.steps, args.warmup) for k, gr in dg.items()}
        best = min(dense_t, key=dense_t.get)
        us_dense = 1e6 * dense_t[best] / (args.steps * n_tok)
        dense_bytes = 3 * elt * H * D + 2 * elt * D
        extras["dense_bf16"] = {"us_per_call": us_dense, "tokens_per_s": 1e6 / us_dense, "form": best,
                                "gbs": dense_bytes / (us_dense * 1e3), "speedup_sparse": us_dense / us_call,
                                "forms_us": {k: 1e6 * v / (args.steps * n_tok) for k, v in dense_t.items()}}
        del ld, dg
        # the tiny fp32 configuration (D=384, H=1024, B=1, 64 tokens, one weight set; its parity against
        # the oracle is in the tests): the latency of one call, L2-resident
        tname = "tiny-f32-D384-H1024"
        tffns = build_ffns(syn.workload_layers(tname, sets=1), dev)
        tx = syn.workload_tokens(tname, 64).to(dev)
        ty = torch.empty_like(tx)
        tg = capture_step(tffns, tx, ty, stream)
        tt = time_graph(tg, stream, args.steps, args.warmup)
        tus = 1e6 * tt / (args.steps * 64)
        extras["tiny_f32"] = {"workload": tname + ": fp32, D=384, H=1024, B=1, 64 tokens, one weight set "
                              "(L2-resident)", "us_per_call": tus, "tokens_per_s": 1e6 / tus,
                              "gpu_launches_per_call": 2}
        del tffns, tg
        # low-rank gate layer, 32 rotated sets: the gate weights (U, V) of all sets are 316 MB,
        # 2.5x the 129 MB L2, so the gate is read from HBM as in a real model's stack of layers
        li = syn.WORKLOADS[LOPA_WORKLOAD]
        lsets = 32
        llayers = syn.workload_layers(LOPA_WORKLOAD, sets=lsets)
        lffns = build_ffns(llayers, dev)
        lx = syn.workload_tokens(LOPA_WORKLOAD).to(dev)
        ly = torch.empty_like(lx)
        lcounts = live_counts(lffns, lx, stream)
        Hp, r = li["H"], li["r"]
        lbytes = sum(elt * r * (D + Hp) + 2 * elt * k * D + 2 * elt * D for k in lcounts)
        lg = capture_step(lffns, lx, ly, stream)
        lt = time_graph(lg, stream, args.steps, args.warmup)
        lus = 1e6 * lt / (args.steps * li["tokens"])
        lgbs = lbytes * args.steps / (lt * 1e9)
        extras["lopa"] = {"workload": LOPA_WORKLOAD, "weight_sets": lsets, "us_per_call": lus,
                          "tokens_per_s": 1e6 / lus, "mean_live": sum(lcounts) / len(lcounts),
                          "gbs": lgbs, "frac_of_measured": lgbs / peak, "frac_of_8tbs": lgbs / NOMINAL_HBM_GBS,
                          "speedup_vs_dense_bf16": us_dense / lus, "gpu_launches_per_call": 3,
                          "flop_ratio_eq4": flops.dense_macs(D, H) /
                          flops.lopa_macs(D, Hp, r, sum(lcounts) / len(lcounts))}
        del lg
        lopa_batched = lopa_batched_extras(lffns, lx, stream, args, peak, D, Hp, r)
        del lffns
        # the low-rank gate with weight-only int8 weights (one scale per row of U, V, W3, W2)
        l8ffns = build_ffns(llayers, dev, dtype="int8")
        l8counts = live_counts(l8ffns, lx, stream)
        l8bytes = sum(r * (D + Hp) + 4 * (r + Hp) + 2 * k * D + 4 * k + 2 * elt * D + 4 * D for k in l8counts)
        l8g = capture_step(l8ffns, lx, ly, stream)
        l8t = time_graph(l8g, stream, args.steps, args.warmup)
        l8us = 1e6 * l8t / (args.steps * li["tokens"])
        extras["lopa_int8_weights"] = {"workload": LOPA_WORKLOAD + ", weight-only int8 (one fp32 scale per row of "
                                       "U, V, W3 and W2), bf16 x and y", "weight_sets": lsets,
                                       "us_per_call": l8us, "tokens_per_s": 1e6 / l8us,
                                       "mean_live": sum(l8counts) / len(l8counts),
                                       "gbs": l8bytes * args.steps / (l8t * 1e9),
                                       "frac_of_measured": l8bytes * args.steps / (l8t * 1e9) / peak,
                                       "speedup_vs_dense_bf16": us_dense / l8us, "gpu_launches_per_call": 3}
        del l8ffns, l8g
        # the pages' complete low-rank form: W1(x) = Gx + U RMSNorm(Vx), double activation
        import activation_sparse_gated_gb300 as sffn_mod
        full = sffn_mod.SFFN_GATE_TILED_G | sffn_mod.SFFN_GATE_RMSNORM | sffn_mod.SFFN_DOUBLE_ACT
        del llayers
        flayers = syn.workload_layers(LOPA_WORKLOAD, sets=lsets, full_form=True)
        fffns = build_ffns(flayers, dev, flags=full)
        fcounts = live_counts(fffns, lx, stream)
        fbytes = sum(elt * r * (D + Hp) + 2 * elt * k * D + 2 * elt * D for k in fcounts)
        fg = capture_step(fffns, lx, ly, stream)
        ft = time_graph(fg, stream, args.steps, args.warmup)
        fus = 1e6 * ft / (args.steps * li["tokens"])
        extras["lopa_full_form"] = {"workload": LOPA_WORKLOAD + " + tiled G, RMSNorm(Vx), double activation",
                                    "weight_sets": lsets, "us_per_call": fus, "tokens_per_s": 1e6 / fus,
                                    "mean_live": sum(fcounts) / len(fcounts),
                                    "gbs": fbytes * args.steps / (ft * 1e9),
                                    "frac_of_measured": fbytes * args.steps / (ft * 1e9) / peak,
                                    "speedup_vs_dense_bf16": us_dense / fus, "gpu_launches_per_call": 3}
        del fffns, fg, flayers
        # the smooth SiLU gate with a live threshold: an unshifted gate (z ~ N(0, 1)),
        # |SiLU(z)| > 1.0 keeps ~10 % of the units; the skip is then an approximation
        slayers = syn.workload_layers(WORKLOAD, sets=n_sets, s=0.5)
        sffns = build_ffns(slayers, dev, act="silu", thr=1.0)
        scounts = live_counts(sffns, x, stream)
        sbytes = sum(elt * H * D + 2 * elt * k * D + 2 * elt * D for k in scounts)
        sg = capture_step(sffns, x, y, stream)
        st = time_graph(sg, stream, args.steps, args.warmup)
        sus = 1e6 * st / (args.steps * n_tok)
        extras["silu_threshold"] = {"workload": WORKLOAD + " with an unshifted gate, SiLU, live iff |A(z)| > 1.0",
                                    "weight_sets": n_sets, "us_per_call": sus, "tokens_per_s": 1e6 / sus,
                                    "mean_live": sum(scounts) / len(scounts),
                                    "gbs": sbytes * args.steps / (st * 1e9),
                                    "frac_of_measured": sbytes * args.steps / (st * 1e9) / peak,
                                    "speedup_vs_dense_bf16": us_dense / sus, "gpu_launches_per_call": 2}
        del sffns, sg, slayers
        # weight-only int8 (per-output-channel scales, quantised on the device), same layers
        qffns = build_ffns(layers, dev, dtype="int8")
        qcounts = live_counts(qffns, x, stream)
        qbytes = sum(H * D + 4 * H + 2 * k * D + 4 * k + 2 * elt * D + 4 * D for k in qcounts)
        qg = capture_step(qffns, x, y, stream)
        qt = time_graph(qg, stream, args.steps, args.warmup)
        qus = 1e6 * qt / (args.steps * n_tok)
        extras["int8_weights"] = {"workload": WORKLOAD + ", weight-only int8 (per-output-channel fp32 scales), "
                                  "bf16 x and y", "weight_sets": n_sets, "us_per_call": qus,
                                  "tokens_per_s": 1e6 / qus, "mean_live": sum(qcounts) / len(qcounts),
                                  "gbs": qbytes * args.steps / (qt * 1e9),
                                  "frac_of_measured": qbytes * args.steps / (qt * 1e9) / peak,
                                  "speedup_vs_dense_bf16": us_dense / qus, "gpu_launches_per_call": 2}
        del qffns, qg
        # weight-only int4 (codes in [-7, 7], two per byte), same layers
        q4ffns = build_ffns(layers, dev, dtype="int4")
        q4counts = live_counts(q4ffns, x, stream)
        q4bytes = sum(H * D // 2 + 4 * H * (D // 64) + k * D + 4 * k * (D // 64) + 2 * elt * D + 4 * D
                      for k in q4counts)
        q4g = capture_step(q4ffns, x, y, stream)
        q4t = time_graph(q4g, stream, args.steps, args.warmup)
        q4us = 1e6 * q4t / (args.steps * n_tok)
        extras["int4_weights"] = {"workload": WORKLOAD + ", weight-only int4 (codes in [-7, 7], two per byte; "
                                  "fp32 scales per 64-column group of W1 and W3, per output channel of W2), "
                                  "bf16 x and y", "weight_sets": n_sets,
                                  "us_per_call": q4us, "tokens_per_s": 1e6 / q4us,
                                  "mean_live": sum(q4counts) / len(q4counts),
                                  "gbs": q4bytes * args.steps / (q4t * 1e9),
                                  "frac_of_measured": q4bytes * args.steps / (q4t * 1e9) / peak,
                                  "speedup_vs_dense_bf16": us_dense / q4us, "gpu_launches_per_call": 2}
        del q4ffns, q4g
        extras["batched"] = batched_extras(ffns, layers, x, stream, args, peak)
        for k, v in lopa_batched.items():  # against the dense standard layer at the same batch (iso-parameter)
            dus = extras["batched"][k]["dense_bf16_us_per_call"]
            v["dense_bf16_us_per_call"] = dus
            v["speedup_vs_dense_bf16"] = dus / v["us_per_call"]
        extras["lopa_batched"] = lopa_batched
        extras["union_skip"] = union_skip_extras(stream, args, peak, dev, "standard", SWEEP_WORKLOAD, 0.95, 4, 4)
        extras["union_skip_lopa"] = union_skip_extras(stream, args, peak, dev, "lopa", LOPA_WORKLOAD, 0.95, 4, 8)

    cpu = None
    if rank == 0 and not args.no_cpu:
        n, dt, cores = time_oracle(layers[:2], x_host, args.cpu_budget, n_tok)
        cpu = {"value": n / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"first {n} tokens of the {WORKLOAD} decode stream (token t through weight set "
                         f"t mod 2), fp64 dense oracle, {dt:.1f} s"}
        one = oracle_one_thread(3.0)
        if one:
            cpu["one_thread"] = one

    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "accumulate": "fp32",
        "data": "synthetic (seeded Gaussian weights, 1/fan-in variance; bias channel shifted for 90% sparsity)",
        "config": {"workload": WORKLOAD, "D": D, "H": H, "B": 1, "tokens_per_step": n_tok,
                   "weight_sets": n_sets, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2: 8 rotated layer sets (881 MB) vs 129 MB L2",
                   "launch": "4096 sffn_forward calls captured in one CUDA graph"},
        "us_per_call": us_call, "us_per_call_eager": us_call_eager, "mean_live_units": mean_live,
        "sparsity": 1 - mean_live / H,
        "hbm": {"gbs": achieved, "frac_of_8tbs": achieved / NOMINAL_HBM_GBS,
                "frac_of_measured": achieved / peak, "bytes_per_call": bytes_step / n_tok},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": ncu_traffic_per_launch(),
                     "peak_source": ("measured copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                                     if peak_kind == "measured" else "fallback 6.8 TB/s"),
                     "kernel": "ffn_b1_bf16_kernel<standard gate>",
                     "algorithmic_bytes_per_launch": bytes_step / n_tok, "kernel_source_hash": kernel_hash()},
        "gpu_launches": args.steps * n_tok * 2,  # forward kernel + finalize kernel per call
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "flop_ratio_eq2": flops.dense_macs(D, H) / flops.sparse_macs(D, H, mean_live),
    }
    out.update(extras)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()


SWEEP_WORKLOAD = "sweep-bf16-D4096-H14336"


def dense_us(ld, x, B, stream, steps, warmup):
    """Dense bf16 FFN via cuBLAS (torch), B tokens per call, call t through set t mod len(ld): the
    faster of the three-GEMM and the concatenated [W1; W3] forms, us per call."""
    import torch
    import torch.nn.functional as F
    calls = x.shape[0] // B
    H = ld[0]["W1"].shape[0]
    y = torch.empty_like(x)
    best = None
    for form in ("three", "concat"):
        def body():
            for t in range(calls):
                L = ld[t % len(ld)]
                xt = x[t * B:(t + 1) * B]
                if form == "three":
                    h = F.relu(F.linear(xt, L["W1"])) * F.linear(xt, L["W3"])
                else:
                    zu = F.linear(xt, L["W13"])
                    h = F.relu(zu[:, :H]) * zu[:, H:]
                y[t * B:(t + 1) * B] = F.linear(h, L["W2"])
        with torch.cuda.stream(stream):
            body()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            body()
        us = 1e6 * time_graph(g, stream, steps, warmup) / (steps * calls)
        best = us if best is None else min(best, us)
        del g
    return best


def set_sparsity(lw, s):
    """Rewrite a layer's bias column (W1[:, D-1], or U[:, r-1] for the low-rank gate) with -Phi^{-1}(s),
    rounded as the generator rounds it (float32, then the storage dtype), on whatever device it lives."""
    import torch
    from activation_sparse_gated_gb300 import synthetic as syn
    W = lw.W1 if lw.r == 0 else lw.U
    col = lw.D - 1 if lw.r == 0 else lw.r - 1
    W[:, col] = torch.tensor(syn.shift_for_sparsity(s), dtype=torch.float32).to(W.dtype).to(W.device)
    return lw


def run_sweep(args):
    """Sparsity x batch sweep at D=4096: standard gate (H=14336) and low-rank gate (H'=19649, r=640),
    s in {0.5, 0.75, 0.9, 0.95}, B in {1, 8, 32, 128}, 1024 tokens per point, each point next to the
    dense bf16 FFN of the standard shape.  One JSON line per point.

    Weight sets: the four generated sets of each gate.  The standard gate rotates four handles (gate
    matrices 470 MB, 3.6x L2).  The low-rank gate matrices of four sets are only 122 MB, so the
    low-rank points rotate sixteen handles (each set loaded into four, every handle a separate copy in
    HBM: 491 MB of gate weights, 3.8x L2).  A sparsity is set by rewriting the bias column (W1[:, D-1]
    or U[:, r-1]) with -Phi^{-1}(s), which gives the same weights as generating the set at that s."""
    import time
    import torch
    import activation_sparse_gated_gb300 as sffn
    from activation_sparse_gated_gb300 import build as libbuild
    from activation_sparse_gated_gb300 import synthetic as syn

    torch.cuda.set_device(0)
    dev = torch.device("cuda:0")
    libbuild.build()
    sffn.load()
    t_start = time.time()
    w = syn.WORKLOADS[SWEEP_WORKLOAD]
    D, H, r, Hp, n_sets = w["D"], w["H"], w["r"], w["Hp"], w["sets"]
    x = syn.workload_tokens(SWEEP_WORKLOAD).to(dev)
    n_tok = x.shape[0]
    stream = torch.cuda.Stream(device=dev)
    peak, _ = measured_peaks()
    elt = 2
    tc_min = int(os.environ.get("SFFN_TC_MIN_BATCH", "2"))
    points = 0
    dense = {}
    for gate in ("standard", "lopa"):
        layers = syn.workload_layers(SWEEP_WORKLOAD, sets=n_sets, gate=gate, s=0.9)
        for lw in layers:
            for k in ("W1", "U", "V", "W3", "W2"):
                if getattr(lw, k) is not None:
                    setattr(lw, k, getattr(lw, k).to(dev))
        if gate == "standard":
            ld = [{"W1": lw.W1, "W3": lw.W3, "W2": lw.W2, "W13": torch.cat([lw.W1, lw.W3], 0)} for lw in layers]
            for B in w["B"]:
                dense[B] = dense_us(ld, x, B, stream, args.steps, args.warmup)
            del ld
        handles = layers if gate == "standard" else layers * 4
        Hg = H if gate == "standard" else Hp
        for s in w["s"]:
            for lw in layers:
                set_sparsity(lw, s)
            ffns = build_ffns(handles, dev)
            torch.cuda.synchronize()
            for B in w["B"]:
                calls = n_tok // B
                y = torch.empty_like(x)
                lives, unions = [], []
                with torch.cuda.stream(stream):
                    for t in range(min(calls, 256)):
                        f = ffns[t % len(ffns)]
                        sffn.sffn_forward(f.h, x[t * B:(t + 1) * B], y[t * B:(t + 1) * B], B, stream)
                        m = f.active_mask(B)
                        lives.append(float(m.sum(axis=1).mean()))
                        unions.append(int(m.any(axis=0).sum()))
                stream.synchronize()
                live, union = sum(lives) / len(lives), sum(unions) / len(unions)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for t in range(calls):
                        sffn.sffn_forward(ffns[t % len(ffns)].h, x[t * B:(t + 1) * B], y[t * B:(t + 1) * B],
                                          B, stream)
                us = 1e6 * time_graph(g, stream, args.steps, args.warmup) / (args.steps * calls)
                del g
                gate_bytes = elt * H * D if gate == "standard" else elt * r * (D + Hp)
                bytes_call = gate_bytes + 2 * elt * union * D + 2 * elt * B * D
                if B == 1:
                    path = "stream kernel" + (" + low-rank t kernel" if gate == "lopa" else "")
                elif B >= tc_min:
                    path = ("tensor cores: gate-up + down kernels (streams every unit slice)" if gate == "standard"
                            else "tensor cores: t pair, gate-up (U t and W3 x) + down kernels")
                else:
                    path = "CUDA cores, union gathers, <= 8 tokens per pass"
                gbs = bytes_call / (us * 1e3)
                print(json.dumps({
                    "sweep": SWEEP_WORKLOAD, "gate": gate, "s": s, "B": B, "D": D, "H": Hg,
                    "r": r if gate == "lopa" else 0, "weight_sets": len(ffns), "path": path,
                    "us_per_call": us, "tokens_per_s": B * 1e6 / us,
                    "measured_sparsity": 1 - live / Hg, "union_fraction": union / Hg,
                    "bytes_per_call": bytes_call, "gbs": gbs, "frac_of_measured": gbs / peak,
                    "dense_bf16_us_per_call": dense[B], "speedup_vs_dense_bf16": dense[B] / us,
                    "dense_bf16_gbs": (3 * elt * H * D + 2 * elt * B * D) / (dense[B] * 1e3)}), flush=True)
                points += 1
            del ffns
            torch.cuda.synchronize()
        del layers, handles
        torch.cuda.empty_cache()
    print(json.dumps({"sweep": SWEEP_WORKLOAD, "points": points, "seconds": time.time() - t_start,
                      "peak_gbs": peak}), flush=True)


PROFILE_CASES = {
    "std": ("std-bf16-D2560-H7168-B1", None),
    "lopa": ("lopa-bf16-D2560-H9787-r400-B1", None),
    "std4096": ("sweep-bf16-D4096-H14336", "standard"),
    "lopa4096": ("sweep-bf16-D4096-H14336", "lopa"),
    "tiny": ("tiny-f32-D384-H1024", None),
}


def run_profile_case(args):
    """A short forward loop for profiler captures: ONE full-size layer of the named
    workload, `--calls` forwards of `--batch` tokens, each followed by a
    synchronisation.  Device memory stays near one layer (110-130 MB at D=2560,
    350 MB at D=4096); the profiler flushes caches between replays, so its DRAM
    figures are cold-cache figures.  Prints one line, times nothing."""
    import torch
    from activation_sparse_gated_gb300 import synthetic as syn
    import activation_sparse_gated_gb300 as sffn
    name, gate = PROFILE_CASES[args.profile_case]
    lw = syn.workload_layers(name, sets=1, gate=gate, **({} if args.sparsity is None else {"s": args.sparsity}))[0]
    dtype = {"int8": "int8", "int4": "int4", "bf16": "bf16", "f32": "f32"}.get(args.dtype or "", lw.dtype)
    ffn = sffn.SparseFFN(lw.D, lw.H, lw.r, "relu", dtype)
    w = {k: (None if t is None else t.cuda()) for k, t in lw.tensors().items()}
    ffn.set_weights(w["W1"] if lw.r == 0 else w["U"], w["V"], w["W3"], w["W2"])
    if args.live_fraction is not None:
        ffn.set_live_fraction_hint(args.live_fraction)
    x = syn.workload_tokens(name, args.calls * args.batch).cuda()
    for c in range(args.calls):
        ffn(x[c * args.batch:(c + 1) * args.batch])
        ffn.synchronize()
    torch.cuda.synchronize()
    print(f"profile case {args.profile_case}: {args.calls} calls of {args.batch} tokens, live units of the "
          f"last call: {ffn.active_counts(args.batch)}", flush=True)


def build_parser() -> argparse.ArgumentParser:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true", help="skip the dense and low-rank comparisons")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of CPU oracle work")
    ap.add_argument("--sweep", action="store_true",
                    help="the D=4096 sparsity x batch sweep (both gates, one JSON line per point) instead of the step")
    ap.add_argument("--profile-case", choices=sorted(PROFILE_CASES), default=None,
                    help="run a short forward loop on one layer of this workload for a profiler capture (no timing)")
    ap.add_argument("--calls", type=int, default=8, help="--profile-case: forwards to run")
    ap.add_argument("--batch", type=int, default=1, help="--profile-case: tokens per forward")
    ap.add_argument("--sparsity", type=float, default=None,
                    help="--profile-case: rewrite the gate's bias for this sparsity (default: the workload's)")
    ap.add_argument("--live-fraction", type=float, default=None,
                    help="--profile-case: the handle's live-fraction hint (picks the kernels of 3..16-token batches)")
    ap.add_argument("--dtype", choices=["bf16", "f32", "int8", "int4"], default=None,
                    help="--profile-case: handle dtype (default: the workload's; int8 / int4 quantise on the device)")
    ap.add_argument("--oracle-one-thread", type=float, default=0.0, metavar="SECONDS",
                    help="(internal) time the oracle on this process's OpenMP threads for SECONDS, print JSON")
    return ap


def main():
    args = build_parser().parse_args()
    args.warmup = max(args.warmup, 3)   # at least three untimed warm-up steps
    if args.oracle_one_thread > 0:
        from activation_sparse_gated_gb300 import synthetic as syn
        n, dt, cores = time_oracle(syn.workload_layers(WORKLOAD, sets=2), syn.workload_tokens(WORKLOAD, 64),
                                   args.oracle_one_thread, 64)
        print(json.dumps({"tokens": n, "seconds": dt, "cores": cores}), flush=True)
        return
    if args.profile_case:
        run_profile_case(args)
    elif args.sweep:
        run_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
