#!/usr/bin/env python3
"""Benchmark of the routed-expert W4A8 MoE layer (one JSON line on rank 0).

A step is one call of the whole layer (route, permute, gate/up projection,
SiLU*up, requant, down projection, combine) on one batch of the decode
workload: T=4 tokens, hidden 2048, 512 routed experts + 1 shared expert,
top-10, intermediate 512, int4 group 128.  Inputs are synthetic and seeded.
The metric is tokens/s of the layer.

L2: the timed steps rotate over 4 device copies of the 857 MB expert bank
and 64 token batches, so each step reads experts that are not in the 129 MB
L2 (the same bytes come back only after >= 3 other banks' steps).

--impl reference times the CPU oracle (test infrastructure, plain C) on the
host cores on a bounded sample of the same workload.

Multi-GPU: the layer needs no exchange between GPUs here; each rank runs an
independent replica on its own batches (weak scaling) and the slowest
rank's time is reported.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

REPO = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, REPO)

WORKLOAD = "decode_t4"
# The headline metric, shared by both arms: tokens/s is the line's value; the HBM (decode) or tensor
# (prefill) throughput against the GPU's peak is its roofline object.
METRIC = "W4A8 MoE layer tokens/s; decode HBM GB/s & prefill i8 TOPS vs GB300 peak"
N_BANKS = 4
N_BATCHES = 64
GRAPH_STEPS = 128
FALLBACK_HBM_GBS = 6800.0


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=200)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=WORKLOAD)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--batches", type=int, default=N_BATCHES, help="token batches rotated between steps")
    p.add_argument("--banks", type=int, default=N_BANKS,
                   help="bank copies rotated between steps (fewer: a smaller case for profiler captures)")
    return p.parse_args()


def _dist_init(n):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    return rank, world


def max_over_ranks(ms: float, world: int, device=None) -> float:
    """The slowest rank's time: every rank gets the same value (all-reduce MAX).

    device: where the reduction tensor lives (a CUDA device for NCCL, None / CPU for gloo).
    """
    if world <= 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, ms_total: float, steps: int) -> float:
    """Units processed by all ranks per second, timed by the slowest rank (weak scaling: fixed units per rank)."""
    return units_per_rank * world * steps / (ms_total * 1e-3)


def _peaks():
    path = os.path.join(REPO, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        for key in ("hbm_gbs", "hbm_GBs", "hbm"):
            if key in pk:
                return float(pk[key]), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _touched_bytes(w, logits_batches):
    """Algorithmic HBM bytes of one step: weights + scales of the touched experts, activations, output."""
    per_expert = (2 * w.I * w.H // 2 + 2 * w.I * (w.H // w.group) * 4 + w.H * w.I // 2 + w.H * (w.I // w.group) * 4)
    tot = []
    for lg in logits_batches:
        ids = np.argsort(-lg, axis=1, kind="stable")[:, :w.top_k]
        experts = len(np.unique(ids)) + w.S
        act = w.T * w.H + 4 * w.T + 4 * w.T * w.E + 4 * w.T * w.H
        tot.append(experts * per_expert + act)
    return float(np.mean(tot)), per_expert


# DRAM traffic per launch of the decode kernel, from an ncu capture of the
# decode workload (dram__bytes_read.sum + dram__bytes_write.sum), valid only
# for the kernel source it was taken on: the file records the SHA-1 of
# csrc/decode.cu at capture time, and a changed kernel reports null.
TRAFFIC_FILE = os.path.join(REPO, "bit_moe_expert_router_gb300", "ncu_traffic.json")


def _decode_traffic(workload: str):
    import hashlib
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f).get("decode_kernel", {})
        with open(os.path.join(REPO, "bit_moe_expert_router_gb300", "csrc", "decode.cu"), "rb") as f:
            sha = hashlib.sha1(f.read()).hexdigest()
    except (OSError, ValueError):
        return None
    if rec.get("source_sha1") != sha or rec.get("workload") != workload:
        return None
    return rec.get("dram_bytes_per_launch")


def run_ours(a):
    import torch
    from bit_moe_expert_router_gb300 import binding, synth

    rank, world = _dist_init(a.gpus)
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS[a.workload]
    d = binding.dims_of(w.T, w.H, w.I, w.E, w.S, w.top_k, w.group)

    bank = synth.make_bank(w)
    bank_mb = sum(x.nbytes for x in (bank.w13, bank.s13, bank.w2, bank.s2)) / 1e6
    banks = []
    for _ in range(a.banks):
        banks.append(tuple(torch.from_numpy(x).to(dev) for x in (bank.w13, bank.s13, bank.w2, bank.s2)))
    batches = [synth.make_tokens(w, batch=rank * a.batches + b) for b in range(a.batches)]
    dev_batches = [tuple(torch.from_numpy(x).to(dev) for x in (t.x_q, t.x_scale, t.logits)) for t in batches]
    ws = binding.alloc_workspace(binding.moe_w4a8_workspace_size(d), dev)
    out = torch.empty((w.T, w.H), dtype=torch.float32, device=dev)
    alg_bytes, per_expert = _touched_bytes(w, [t.logits for t in batches])
    engine = binding.moe_w4a8_engine_for(d)
    kernel_label = {binding.ENGINE_DECODE: "decode_kernel (fused, one launch per step; timed with its barrier memset)",
                    binding.ENGINE_TCGEN05: "whole step (9 kernels of the tcgen05 engine)",
                    binding.ENGINE_GROUPED: "whole step (7 kernels of the grouped engine)"}[engine]
    launches_per_step = {binding.ENGINE_DECODE: 1, binding.ENGINE_TCGEN05: 9, binding.ENGINE_GROUPED: 7}[engine]

    def step(i):
        x_q, x_s, lg = dev_batches[i % len(dev_batches)]
        w13, s13, w2, s2 = banks[i % len(banks)]
        binding.moe_w4a8_forward(x_q, x_s, lg, w13, s13, w2, s2, d, out, ws)

    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        for i in range(max(a.warmup, 3)):
            step(i)
    torch.cuda.synchronize(dev)

    # capture GRAPH_STEPS consecutive steps; replay to cover exactly K steps
    g_full = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_full, stream=stream):
        for i in range(GRAPH_STEPS):
            step(i)
    rem = a.steps % GRAPH_STEPS
    g_rem = None
    if rem:
        g_rem = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_rem, stream=stream):
            for i in range(rem):
                step(i)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        g_full.replay()
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    if rank == 0:
        clocks.start()
        time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(a.steps // GRAPH_STEPS):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    clk = clocks.stop() if rank == 0 else None
    ms_per_step = ms / a.steps

    # plain launches (no graph), same stream, for the launch-overhead picture
    n_plain = min(a.steps, 2000)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(n_plain):
            step(i)
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    plain_ms_per_step = ev0.elapsed_time(ev1) / n_plain

    # end to end through the public API: the step's inputs start in pinned host memory and its
    # output ends there (moe_w4a8_forward_host: one kernel reads the inputs over the host link into
    # the workspace, the layer writes the output into host memory), every step
    host_in = [tuple(torch.from_numpy(x).pin_memory() for x in (t.x_q, t.x_scale, t.logits)) for t in batches]
    host_out = torch.empty((w.T, w.H), dtype=torch.float32).pin_memory()
    ws_host = binding.alloc_workspace(binding.moe_w4a8_forward_host_workspace_size(d), dev)
    n_e2e = min(a.steps, 2000)

    def e2e_step(i):
        x_q, x_scale, logits = host_in[i % len(host_in)]
        w13, s13, w2, s2 = banks[i % len(banks)]
        binding.moe_w4a8_forward_host(x_q, x_scale, logits, w13, s13, w2, s2, d, host_out, ws_host)

    with torch.cuda.stream(stream):
        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for i in range(n_e2e):
            e2e_step(i)
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = ev0.elapsed_time(ev1) / n_e2e
    h2d = sum(x.numel() * x.element_size() for x in host_in[0])
    d2h = host_out.numel() * host_out.element_size()

    if rank != 0:
        return
    peak, peak_kind = _peaks()
    achieved = alg_bytes / (ms_per_step * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": whole_job_rate(w.T, world, ms, a.steps),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": a.steps,
        "warmup": a.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int8",
        "data": "synthetic (seeded generator: bf16 N(0,1) activations -> int8, N(0,0.02) weights -> int4 g128)",
        "config": {"workload": w.name, "T": w.T, "H": w.H, "I": w.I, "E": w.E, "n_shared": w.S, "top_k": w.top_k,
                   "group": w.group, "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: {len(banks)} bank copies x {bank_mb:.0f} MB and {len(batches)} token batches rotated",
                   "timing": f"CUDA graph of {GRAPH_STEPS} steps replayed; events on the launching stream"},
        "plain_launch_ms_per_step": plain_ms_per_step,
        "e2e": {"value": w.T / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "call": "moe_w4a8_forward_host on pinned host buffers (inputs staged by one kernel, output written in place)"},
        "gpu_launches": a.steps * launches_per_step,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": _decode_traffic(w.name) if engine == binding.ENGINE_DECODE else None,
                     "peak_source": peak_kind,
                     "kernel": kernel_label, "algorithmic_bytes_per_step": alg_bytes,
                     "bytes_per_touched_expert": per_expert},
        "clocks": clk,
    }
    if not a.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=12.0)
    print(json.dumps(line), flush=True)


def cpu_baseline(w, budget_s: float):
    """The oracle as it stands on the host cores, on a bounded sample of token batches."""
    import oracle
    from bit_moe_expert_router_gb300 import synth
    bank = synth.make_bank(w)
    toks, t0, n = 0, time.perf_counter(), 0
    while True:
        tok = synth.make_tokens(w, batch=1000 + n)
        oracle.forward_workload(w, tok, bank)
        toks += w.T
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    cores = min(os.cpu_count() or 1, w.T, int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1)))
    return {"value": toks / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} batches of T={w.T} tokens of {w.name} ({toks} tokens, {el:.1f} s; threads over tokens)"}


def run_reference(a):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from bit_moe_expert_router_gb300 import synth
    import oracle
    import numpy as np
    w = synth.WORKLOADS[a.workload]
    bank = synth.make_bank(w)
    # warm-up on whole batches, which also measures the oracle's time per token
    t_tok = None
    for b in range(max(a.warmup, 1)):
        t0 = time.perf_counter()
        oracle.forward_workload(w, synth.make_tokens(w, batch=b), bank)
        t_tok = (time.perf_counter() - t0) / w.T
    # exactly a.steps steps; each step is a sample of the step's batch (its first n_tok tokens),
    # sized so that the timed steps take about two minutes at most
    n_tok = int(max(1, min(w.T, 120.0 / (a.steps * max(t_tok, 1e-9)))))
    el = 0.0
    for b in range(a.steps):
        tok = synth.make_tokens(w, batch=max(a.warmup, 1) + b)
        t0 = time.perf_counter()
        oracle.forward_workload(w, tok, bank, np.arange(n_tok))
        el += time.perf_counter() - t0
    ms = el * 1e3 / a.steps
    val = n_tok / (ms * 1e-3)
    cores = min(os.cpu_count() or 1, n_tok)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
        "n_gpus": 1, "steps": a.steps, "warmup": a.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "H": w.H, "I": w.I, "E": w.E, "n_shared": w.S, "top_k": w.top_k,
                   "group": w.group, "parallelism": "cpu"},
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{a.steps} steps of {n_tok} of the T={w.T} tokens of a batch of {w.name}"},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    a = _args()
    import __graft_entry__
    __graft_entry__.build()
    if a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)


if __name__ == "__main__":
    main()
