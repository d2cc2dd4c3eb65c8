#!/usr/bin/env python3
"""Benchmark of the routed-expert W4A8 MoE layer (one JSON line on rank 0).

A step is one call of the whole layer (route, permute, gate/up projection,
SiLU*up, requant, down projection, combine) through moe_w4a8_forward on one
batch of synthetic, seeded input.  The headline line is the decode workload
(T=4 tokens, hidden 2048, 512 routed experts + 1 shared, top-10,
intermediate 512, int4 group 128): tokens/s of the layer and its HBM
roofline.  The same run also times the other three workloads of the layer
(draft verification T=12, prefill T=8192, the 288-expert bank T=2048) for the
same K steps and reports each under "workloads" with its own roofline: HBM
bytes of the touched experts for the decode batches, integer multiply-adds
on the tensor cores for prefill, and max(bytes / bandwidth, ops / tensor
peak) for the large bank, which sits near the ridge.

Timing: each workload's K steps are captured in a CUDA graph and the K-step
region is replayed R times, each replay bracketed by CUDA events on the
launching stream; the reported time is the median region (spread given).

L2: decode steps rotate over 4 device copies of the 857 MB expert bank and
64 token batches, so each step reads experts that are not in the 129 MB L2;
the prefill and large-bank steps stream banks of 857 MB and 2.9 GB that do
not fit it.

--impl reference times the CPU oracle (test infrastructure, plain C) on the
host cores on a bounded sample of the same workload.

Multi-GPU: the layer needs no exchange between GPUs here; each rank runs an
independent replica on its own batches (weak scaling) and the slowest
rank's time is reported.
"""
from __future__ import annotations

import argparse
import hashlib
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
# Further workloads timed in the same run (reported under "workloads").
EXTRA_WORKLOADS = ("decode_verify_t12", "prefill_t8192", "large_bank_t2048")
# The headline metric, shared by both arms: tokens/s is the line's value; the HBM (decode) or tensor
# (prefill) throughput against the GPU's peak is its roofline object.
METRIC = "W4A8 MoE layer tokens/s; decode HBM GB/s & prefill i8 TOPS vs GB300 peak"
N_BANKS = 4
N_BATCHES = 64
GRAPH_STEPS = 128
REPEATS = 15
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

# DRAM traffic per launch of the decode kernel, from an ncu capture of the
# decode workload (dram__bytes_read.sum + dram__bytes_write.sum), valid only
# for the kernel source it was taken on: the record names the SHA-1 of
# csrc/decode.cu at capture time, and a changed kernel reports null.
TRAFFIC_FILE = os.path.join(REPO, "profiles", "ncu_traffic.json")


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=WORKLOAD)
    p.add_argument("--only", action="store_true", help="time the named workload alone (no further workloads)")
    p.add_argument("--repeats", type=int, default=REPEATS, help="replays of the K-step region (median reported)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--batches", type=int, default=N_BATCHES, help="token batches rotated between decode steps")
    p.add_argument("--banks", type=int, default=N_BANKS,
                   help="bank copies rotated between decode steps (fewer: a smaller case for profiler captures)")
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


def peaks():
    """(HBM GB/s, dense bf16 TFLOP/s burst, sustained, source) from the measured peaks file, else the fallback."""
    path = os.path.join(REPO, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        hbm = float(pk["hbm_gbs"])
        tf = float(pk["bf16_tflops"])
        tfs = float(pk.get("bf16_tflops_sustained", tf))
        return hbm, tf, tfs, "measured"
    except (OSError, ValueError, KeyError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS, "fallback"


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
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        # "under load": samples drawing more than the idle power
        loaded = [s for s, p in zip(sm, power) if p > 1.5 * min(power)] if power else []
        return {"sm_mhz": statistics.median(loaded or sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons), "samples": len(sm),
                "samples_under_load": len(loaded)}


def per_expert_bytes(w) -> int:
    """Weights + scales of one expert (both projections)."""
    return (2 * w.I * w.H // 2 + 2 * w.I * (w.H // w.group) * 4 + w.H * w.I // 2 + w.H * (w.I // w.group) * 4)


def touched_bytes(w, logits_batches):
    """Algorithmic HBM bytes of one step: weights + scales of the touched experts, activations, logits, output."""
    tot = []
    for lg in logits_batches:
        ids = np.argsort(-lg, axis=1, kind="stable")[:, :w.top_k]
        experts = len(np.unique(ids)) + w.S
        act = w.T * w.H + 4 * w.T + 4 * w.T * w.E + 4 * w.T * w.H
        tot.append(experts * per_expert_bytes(w) + act)
    return float(np.mean(tot))


def touched_bytes_mixed(w, logits_batches, slot_bits):
    """touched_bytes for a bank whose 2-bit slots (slot_bits[e] == 2) are stored 4 codes per byte: such a
    slot's code bytes halve, its scales stay."""
    codes = w.H * (2 * w.I) // 2 + w.I * w.H // 2
    tot = []
    for lg in logits_batches:
        ids = np.argsort(-lg, axis=1, kind="stable")[:, :w.top_k]
        slots = list(np.unique(ids)) + [w.E + s for s in range(w.S)]
        two = sum(1 for e in slots if slot_bits[e] == 2)
        act = w.T * w.H + 4 * w.T + 4 * w.T * w.E + 4 * w.T * w.H
        tot.append(len(slots) * per_expert_bytes(w) - two * codes // 2 + act)
    return float(np.mean(tot))


def step_ops(w) -> float:
    """Integer multiply-adds of one step counted as 2 ops each: every pair row's gate/up and down projections."""
    return float(w.pairs) * 2.0 * (2 * w.I * w.H + w.H * w.I)


def decode_traffic(workload: str):
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


def time_region(step, steps, repeats, stream, dev):
    """Median, min and max of `repeats` replays of a CUDA graph of exactly `steps` consecutive steps (ms)."""
    import torch
    graphs = []
    done = 0
    while done < steps:
        n = min(GRAPH_STEPS, steps - done)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                step(done + i)
        graphs.append(g)
        done += n
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        for g in graphs:
            g.replay()
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(repeats):
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for g in graphs:
                g.replay()
            ev1.record(stream)
        torch.cuda.synchronize(dev)
        times.append(ev0.elapsed_time(ev1))
    return statistics.median(times), min(times), max(times)


def run_ours(a):
    import torch
    from bit_moe_expert_router_gb300 import binding, synth

    rank, world = _dist_init(a.gpus)
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    hbm_peak, tf_peak, tf_sustained, peak_kind = peaks()

    bank_cache, host_banks = {}, {}

    def host_bank(w):
        key = (w.H, w.I, w.E, w.S, w.group, w.twobit_frac, w.seed)
        if key not in host_banks:
            host_banks[key] = synth.make_bank(w)
        return host_banks[key]

    def device_banks(w, copies):
        key = (w.H, w.I, w.E, w.S, w.group, w.twobit_frac, w.seed)
        have = bank_cache.get(key, [])
        if len(have) < copies:
            bank = host_bank(w)
            while len(have) < copies:
                have.append(tuple(torch.from_numpy(x).to(dev) for x in (bank.w13, bank.s13, bank.w2, bank.s2)))
            bank_cache[key] = have
        return have[:copies]

    def measure(name, n_banks, n_batches, warmup):
        w = synth.WORKLOADS[name]
        d = binding.dims_of(w.T, w.H, w.I, w.E, w.S, w.top_k, w.group)
        banks = device_banks(w, n_banks)
        batches = [synth.make_tokens(w, batch=rank * n_batches + b) for b in range(n_batches)]
        dev_batches = [tuple(torch.from_numpy(x).to(dev) for x in (t.x_q, t.x_scale, t.logits)) for t in batches]
        ws = binding.alloc_workspace(binding.moe_w4a8_workspace_size(d), dev)
        out = torch.empty((w.T, w.H), dtype=torch.float32, device=dev)

        def step(i):
            x_q, x_s, lg = dev_batches[i % len(dev_batches)]
            w13, s13, w2, s2 = banks[i % len(banks)]
            binding.moe_w4a8_forward(x_q, x_s, lg, w13, s13, w2, s2, d, out, ws)

        with torch.cuda.stream(stream):
            for i in range(max(warmup, 3)):
                step(i)
        torch.cuda.synchronize(dev)
        return w, d, banks, batches, step, ws

    # ---------------------------------------------------------------- headline workload
    w, d, banks, batches, step, _ = measure(a.workload, a.banks, a.batches, a.warmup)
    engine = binding.moe_w4a8_engine_for(d)
    launches_per_step = {binding.ENGINE_DECODE: 1, binding.ENGINE_TCGEN05: 10, binding.ENGINE_GROUPED: 8}[engine]
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    if rank == 0:
        clocks.start()
        time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    ms, ms_min, ms_max = time_region(step, a.steps, a.repeats, stream, dev)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    ms = max_over_ranks(ms, world, dev)
    ms_per_step = ms / a.steps
    headline = _roofline_entry(w, ms_per_step, [t.logits for t in batches], hbm_peak, tf_peak, peak_kind, engine,
                               binding)
    if engine == binding.ENGINE_DECODE:
        headline["roofline"]["traffic"] = decode_traffic(w.name)

    # plain launches (no graph), same stream, for the launch-overhead picture
    n_plain = min(a.steps, 2000)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(n_plain):
            step(i)
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    plain_ms_per_step = ev0.elapsed_time(ev1) / n_plain

    e2e = None
    if not a.no_e2e:
        e2e = _e2e(w, d, banks, batches, a.steps, stream, dev, binding)
    # the same workload with each batch's routing supplied (an expert-routing cache hit)
    supplied = _supplied_routing_entry(w, d, banks, batches, a, stream, dev, binding, world)

    # ---------------------------------------------------------------- further workloads, same K steps
    extra = {}
    if not a.only:
        for name in EXTRA_WORKLOADS:
            if name == w.name:
                continue
            wx = synth.WORKLOADS[name]
            decode_like = wx.T <= 32
            wx, dx, _, bx, stepx, wsx = measure(name, a.banks if decode_like else 1,
                                                a.batches if decode_like else 2, a.warmup)
            engx = binding.moe_w4a8_engine_for(dx)
            msx, mnx, mxx = time_region(stepx, a.steps, a.repeats, stream, dev)
            msx = max_over_ranks(msx, world, dev)
            ent = _roofline_entry(wx, msx / a.steps, [t.logits for t in bx], hbm_peak, tf_peak, peak_kind, engx,
                                  binding)
            ent["tokens_per_s"] = whole_job_rate(wx.T, world, msx, a.steps)
            ent["region_ms"] = {"median": msx, "min": mnx, "max": mxx, "repeats": a.repeats}
            ent["config"] = _config(wx, world)
            if wx.twobit_frac > 0:
                ent["mixed_2bit_storage"] = _mixed_entry(wx, dx, bx, stepx, a, stream, dev, binding, world)
            extra[name] = ent
            del wsx
            torch.cuda.empty_cache()

    # the clock samples span every timed region (the idle gaps between them are left out by power)
    clk = clocks.stop() if rank == 0 else None
    if rank != 0:
        return
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
        "config": dict(_config(w, world),
                       l2=f"inputs larger than L2: {len(banks)} bank copies of the expert bank and "
                          f"{len(batches)} token batches rotated",
                       timing=f"CUDA graph of the K steps replayed {a.repeats} times, events on the launching "
                              f"stream, median region reported"),
        "region_ms": {"median": ms, "min": ms_min, "max": ms_max, "repeats": a.repeats},
        "plain_launch_ms_per_step": plain_ms_per_step,
        "gpu_launches": a.steps * launches_per_step,
        "roofline": headline["roofline"],
        "clocks": clk,
    }
    if e2e is not None:
        line["e2e"] = e2e
    line["routing_supplied"] = supplied
    if extra:
        line["workloads"] = extra
    if not a.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=10.0, bank=host_bank(w))
        for name, ent in extra.items():
            wx = synth.WORKLOADS[name]
            ent["cpu_baseline"] = cpu_baseline(wx, budget_s=4.0, bank=host_bank(wx))
    print(json.dumps(line), flush=True)


def _config(w, world):
    return {"workload": w.name, "T": w.T, "H": w.H, "I": w.I, "E": w.E, "n_shared": w.S, "top_k": w.top_k,
            "group": w.group, "parallelism": f"replicas x{world}"}


def _roofline_entry(w, ms_per_step, logits_batches, hbm_peak, tf_peak, peak_kind, engine, binding):
    """Roofline of one step: HBM-bound (decode batches), tensor-bound (prefill) or the larger of the two."""
    alg_bytes = touched_bytes(w, logits_batches)
    ops = step_ops(w)
    t = ms_per_step * 1e-3
    gbs = alg_bytes / t / 1e9
    tops = ops / t / 1e12
    t_hbm = alg_bytes / (hbm_peak * 1e9)
    t_tc = ops / (tf_peak * 1e12)
    engine_name = {binding.ENGINE_DECODE: "decode", binding.ENGINE_TCGEN05: "tcgen05",
                   binding.ENGINE_GROUPED: "grouped"}[engine]
    kernel = ("decode_kernel (fused, one launch per step)" if engine == binding.ENGINE_DECODE
              else f"whole step ({engine_name} engine, all kernels of the call)")
    if t_hbm >= t_tc:
        roof = {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak}
    else:
        roof = {"bound": "tensor", "achieved": tops, "peak": tf_peak, "unit": "TFLOP/s", "frac": tops / tf_peak,
                "mma": "tcgen05.mma kind::f16 (int4 / int8 values exact in fp16, fp32 accumulator); peak = "
                       "measured dense bf16 burst (fp16 runs at the bf16 rate)"}
    roof.update({"traffic": None, "peak_source": peak_kind, "kernel": kernel,
                 "algorithmic_bytes_per_step": alg_bytes, "ops_per_step": ops,
                 "hbm_GBs": gbs, "hbm_frac": gbs / hbm_peak, "tensor_TOPs": tops, "tensor_frac": tops / tf_peak,
                 "roofline_ms": max(t_hbm, t_tc) * 1e3, "roofline_frac": max(t_hbm, t_tc) / t})
    return {"ms_per_step": ms_per_step, "engine": engine_name, "roofline": roof}


def _supplied_routing_entry(w, d, banks, batches, a, stream, dev, binding, world):
    """moe_w4a8_forward_routed with each batch's routing computed once beforehand (moe_w4a8_route, outside the
    timed region): the step without its top-k, as a routing cache would serve it."""
    import torch
    dev_batches = [tuple(torch.from_numpy(x).to(dev) for x in (t.x_q, t.x_scale, t.logits)) for t in batches]
    ws = binding.alloc_workspace(binding.moe_w4a8_workspace_size(d), dev)
    routes = []
    for x_q, x_s, lg in dev_batches:
        ids = torch.empty((w.T, w.top_k), dtype=torch.int32, device=dev)
        wts = torch.empty((w.T, w.top_k), dtype=torch.float32, device=dev)
        ex = [torch.empty(n, dtype=torch.int32, device=dev) for n in (w.E, w.E + 1, w.T * w.top_k, w.T * w.top_k)]
        binding.moe_w4a8_route(lg, d, ids, wts, *ex, ws)
        routes.append((ids, wts))
    out = torch.empty((w.T, w.H), dtype=torch.float32, device=dev)

    def step(i):
        x_q, x_s, _ = dev_batches[i % len(dev_batches)]
        ids, wts = routes[i % len(routes)]
        w13, s13, w2, s2 = banks[i % len(banks)]
        binding.moe_w4a8_forward_routed(x_q, x_s, ids, wts, w13, s13, w2, s2, d, out, ws)

    with torch.cuda.stream(stream):
        for i in range(max(a.warmup, 3)):
            step(i)
    torch.cuda.synchronize(dev)
    ms, mn, mx = time_region(step, a.steps, a.repeats, stream, dev)
    ms = max_over_ranks(ms, world, dev)
    return {"ms_per_step": ms / a.steps, "value": whole_job_rate(w.T, world, ms, a.steps), "unit": "tokens/s",
            "call": "moe_w4a8_forward_routed (routing of each batch computed beforehand by moe_w4a8_route)",
            "region_ms": {"median": ms, "min": mn, "max": mx, "repeats": a.repeats}}


def _mixed_entry(w, d, batches, step_int4, a, stream, dev, binding, world):
    """The same workload with its 2-bit experts stored 4 codes per byte in compact storage (every slot's
    rows at the slot's own width, moe_w4a8_forward_w2w4_compact): time, algorithmic bytes and bank size
    beside the int4 storage's (the same codes)."""
    import torch
    from bit_moe_expert_router_gb300 import synth
    b2 = synth.make_bank(w, pack2=True)
    w13c, o13, w2c, o2 = synth.compact_bank(b2)
    bank = tuple(torch.from_numpy(x).to(dev) for x in (w13c, o13, b2.s13, w2c, o2, b2.s2))
    bits = torch.from_numpy(b2.slot_bits).to(dev)
    dev_batches = [tuple(torch.from_numpy(x).to(dev) for x in (t.x_q, t.x_scale, t.logits)) for t in batches]
    ws = binding.alloc_workspace(binding.moe_w4a8_workspace_size(d), dev)
    out = torch.empty((w.T, w.H), dtype=torch.float32, device=dev)

    def step(i):
        x_q, x_s, lg = dev_batches[i % len(dev_batches)]
        binding.moe_w4a8_forward_w2w4_compact(x_q, x_s, lg, *bank, bits, d, out, ws)

    with torch.cuda.stream(stream):
        for i in range(max(a.warmup, 3)):
            step(i)
    torch.cuda.synchronize(dev)
    ms, mn, mx = time_region(step, a.steps, a.repeats, stream, dev)
    ms = max_over_ranks(ms, world, dev)
    lgs = [t.logits for t in batches]
    scales = int(b2.s13.nbytes + b2.s2.nbytes)
    return {"ms_per_step": ms / a.steps, "algorithmic_bytes_per_step": touched_bytes_mixed(w, lgs, b2.slot_bits),
            "int4_storage_bytes_per_step": touched_bytes(w, lgs),
            "bank_bytes": int(w13c.nbytes + w2c.nbytes) + scales,
            "int4_storage_bank_bytes": int(b2.w13.nbytes + b2.w2.nbytes) + scales,
            "storage": "compact: every slot's rows at the slot's own width (2-bit rows K/4 bytes), slots back "
                       "to back; one bank copy (the int4 line rotates copies to stay beyond L2)",
            "region_ms": {"median": ms, "min": mn, "max": mx, "repeats": a.repeats}}


def _e2e(w, d, banks, batches, steps, stream, dev, binding):
    """End to end through the public API: the step's inputs start in pinned host memory and its output ends
    there (moe_w4a8_forward_host: one kernel reads the inputs over the host link into the workspace, the layer
    writes the output into host memory), every step."""
    import torch
    host_in = [tuple(torch.from_numpy(x).pin_memory() for x in (t.x_q, t.x_scale, t.logits)) for t in batches]
    host_out = torch.empty((w.T, w.H), dtype=torch.float32).pin_memory()
    ws_host = binding.alloc_workspace(binding.moe_w4a8_forward_host_workspace_size(d), dev)
    n_e2e = min(steps, 2000)

    def e2e_step(i):
        x_q, x_scale, logits = host_in[i % len(host_in)]
        w13, s13, w2, s2 = banks[i % len(banks)]
        binding.moe_w4a8_forward_host(x_q, x_scale, logits, w13, s13, w2, s2, d, host_out, ws_host)

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
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
    return {"value": w.T / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": n_e2e,
            "call": "moe_w4a8_forward_host on pinned host buffers (inputs staged by one kernel, output written "
                    "in place)"}


def cpu_baseline(w, budget_s: float, bank=None):
    """The oracle as it stands on the host cores, on a bounded sample of tokens of the workload."""
    import oracle
    from bit_moe_expert_router_gb300 import synth
    if bank is None:
        bank = synth.make_bank(w)
    toks, el, n = 0, 0.0, 0
    # whole batches for small T; otherwise growing token subsets of one batch
    while el < budget_s:
        tok = synth.make_tokens(w, batch=1000 + n)
        sub = None if w.T <= 64 else np.arange(min(w.T, 16 * (n + 1)))
        t0 = time.perf_counter()
        oracle.forward_workload(w, tok, bank, sub)
        el += time.perf_counter() - t0
        toks += w.T if sub is None else len(sub)
        n += 1
    cores = min(os.cpu_count() or 1, int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1)))
    return {"value": toks / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{toks} tokens of {w.name} in {n} calls ({el:.1f} s; threads over tokens)"}


def run_reference(a):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from bit_moe_expert_router_gb300 import synth
    import oracle
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
