#!/usr/bin/env python
"""Benchmark of the GDN slot-pool layer on one GB300 (replicas on N GPUs).

Headline: batched decode at m = 256 active slots of a 256-slot pool, on a
Qwen3.5-35B-A3B-shaped GDN layer (16 q/k heads, 32 v heads, d_k = d_v = 128,
conv width 4, bf16 io, fp32 state ~ N(0, 0.1)), new random inputs every step:
slot-steps/s.  One step is one decode launch over the 256 slots (conv + SiLU,
L2 norms, gates, delta-rule update of every head's state in place, gated
RMSNorm).  The 537 MB of state read and written per step is far larger than
L2, so no flush is needed between steps.

Also reported on the same line: the decode m-sweep {1,4,8,16,64,256}, the
varlen prefill of 8 sequences {1,17,300,4095,1024,2048,513,8000} (tok/s), the
end-to-end number through the public API with host buffers, the roofline of
the decode kernel, the fp64 CPU oracle as a baseline, and the SM clocks seen.

--impl reference times the fp64 CPU oracle on the host cores for the same metric.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

HQK, HV, D, W = 16, 32, 128, 4
C = 2 * HQK * D + HV * D
NUM_SLOTS = 256
M_HEAD = 256
SWEEP = [1, 4, 8, 16, 64, 256]
PREFILL_LENGTHS = [1, 17, 300, 4095, 1024, 2048, 513, 8000]
WORKLOAD_DECODE, WORKLOAD_PREFILL = 2, 3
METRIC = "GDN decode slot-steps/s @m=256"
UNIT = "slot-steps/s"
HEAD_WORKLOAD = ("decode m=256: Qwen3.5-35B-A3B-shaped GDN layer (Hqk 16, Hv 32, d 128, conv 4), "
                 "bf16 io, fp32 state, 256-slot pool, new random inputs each step")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ----------------------------------------------------------- algorithmic bytes ----

def decode_bytes_per_slot_step(io=2):
    """HBM bytes one slot-step must move: S read + write (fp32), conv buffer read (W-1 rows) and one new
    row written, q/k/v/z/a/b read, out written (io dtype)."""
    s = HV * D * D * 4 * 2
    conv = (W - 1) * C * io + C * io
    inputs = C * io + HV * D * io + 2 * HV * io
    out = HV * D * io
    return s + conv + inputs + out


# algorithmic flops per prefill token of the chunked form (64-token chunks, triangular halves):
# K K^T 8 064 + Q K^T 8 320 + solve C^2/3 + W, U, intra-chunk O 3 x 8 320 + 3 state products 3 x 2 d^2,
# times Hv
PREFILL_FLOPS_PER_TOKEN = 4.51e6


def decode_param_bytes():
    return C * W * 4 + 2 * HV * 4 + D * 4


def prefill_bytes(lengths, io=2):
    """Per token: q, k, v, z, a, b in and out; per sequence: S read + write and the conv buffer read + write."""
    T = sum(lengths)
    per_tok = C * io + HV * D * io + 2 * HV * io + HV * D * io
    per_seq = HV * D * D * 4 * 2 + 2 * (W - 1) * C * io
    return T * per_tok + len(lengths) * per_seq + decode_param_bytes()


# ------------------------------------------------------- profiled traffic ----

DECODE_SOURCES = ["gated_deltanet_linear_rule_gb300/csrc/gdn_decode.cu",
                  "gated_deltanet_linear_rule_gb300/csrc/gdn_internal.cuh"]
PREFILL_SOURCES = ["gated_deltanet_linear_rule_gb300/csrc/gdn_chunk.cu",
                   "gated_deltanet_linear_rule_gb300/csrc/gdn_prefill.cu",
                   "gated_deltanet_linear_rule_gb300/csrc/gdn_internal.cuh",
                   "gated_deltanet_linear_rule_gb300/csrc/gdn_tcgen05.cuh"]


def sources_sha256(paths):
    import hashlib

    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic(kernel: str, sources, units: float):
    """DRAM bytes per launch from a committed ncu summary (profiles/*.md) of this kernel, scaled from the
    captured launch's units to `units`; None when no summary matches the current source hash."""
    want = sources_sha256(sources)
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    for name in sorted(os.listdir(pdir)):
        if not name.endswith(".md"):
            continue
        meta = {}
        for line in open(os.path.join(pdir, name)):
            if line.startswith("    ") and ":" in line:
                k, v = line.strip().split(":", 1)
                meta[k.strip()] = v.strip()
        if meta.get("kernel") == kernel and meta.get("source_sha256") == want:
            try:
                return float(meta["dram_bytes_per_launch"]) * units / float(meta["units_per_launch"])
            except (KeyError, ValueError):
                return None
    return None


# -------------------------------------------------------------- clocks ----

class ClockSampler:
    """nvidia-smi samples during the timed region (clocks and throttle reasons)."""

    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
            if self.uuid:
                cmd += ["-i", self.uuid]
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 10:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[6:10]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------- ranks ----

def dist_init():
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return rank, world, local


def reduce_max(x: float, world: int) -> float:
    """Max of a per-rank float over all ranks (the slowest rank sets the job's time)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ----------------------------------------------------------------- GPU arm ----

def make_decode_pool(torch, binding, synth, out_dtype="bf16"):
    pool = binding.Pool(HQK, HV, D, D, NUM_SLOTS, 1, W, "bf16", out_dtype)
    p = synth.layer_params(WORKLOAD_DECODE, 0, HQK, HV, D, D, W)
    pool.layer_params(0, *(torch.from_numpy(p[k]) for k in ("conv_w", "A_log", "dt_bias", "norm_w")))
    for _ in range(NUM_SLOTS):
        pool.alloc()
    g = torch.Generator(device="cuda")
    g.manual_seed(20260)
    block = pool.state_block(0)
    block.copy_(torch.randn(block.shape, generator=g, device="cuda") * math.sqrt(0.1))
    torch.cuda.synchronize()
    return pool


def device_inputs(torch, m, n_sets, seed):
    """n_sets distinct input sets of m rows, N(0, 1) rounded to bf16 (one draw per tensor kind)."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    widths = {"q": HQK * D, "k": HQK * D, "v": HV * D, "z": HV * D, "a": HV, "b": HV}
    full = {n: torch.randn((n_sets, m, w), generator=g, device="cuda").to(torch.bfloat16) for n, w in widths.items()}
    return [{n: full[n][i] for n in widths} for i in range(n_sets)]


def slot_groups(torch, pool, synth, m):
    """Slot-pointer arrays of the 256 // m disjoint groups of m slots of the pool (random order).  A
    timed loop at m slots takes the groups in turn, one per step, so that at small m the states a
    step reads were last touched 256 // m - 1 steps earlier, with (256 - m) x 2.1 MB of other states
    in between -- more than the 129 MB L2 -- and come from HBM, as the whole 256-slot pool does."""
    perm = synth.distinct_slots(WORKLOAD_DECODE, NUM_SLOTS, NUM_SLOTS, sub=m)
    groups = [perm[i * m:(i + 1) * m] for i in range(NUM_SLOTS // m)]
    return [pool.slot_ptrs(0, torch.tensor(g, dtype=torch.int32, device="cuda")) for g in groups]


def time_decode(torch, pool, synth, m, steps, warmup, seed=1):
    """Device time of `steps` back-to-back decode launches at m slots (events on the launching
    stream around the whole region), each step on the next of the pool's disjoint m-slot groups:
    (ms per step, ms per launch, ms per launch)."""
    groups = slot_groups(torch, pool, synth, m)
    n_sets = min(steps + warmup, 200)
    sets = device_inputs(torch, m, n_sets, seed)
    out = torch.empty((m, HV * D), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    for i in range(warmup):
        s = sets[i % n_sets]
        ptrs = groups[i % len(groups)]
        pool.decode_step(0, ptrs, m, s["q"], s["k"], s["v"], s["a"], s["b"], s["z"], out, stream)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push(f"decode_timed_m{m}")
    t0.record(stream)
    for i in range(steps):
        s = sets[(warmup + i) % n_sets]
        ptrs = groups[(warmup + i) % len(groups)]
        pool.decode_step(0, ptrs, m, s["q"], s["k"], s["v"], s["a"], s["b"], s["z"], out, stream)
    t1.record(stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    assert pool.device_status() == 0
    # the launches run back to back: their average duration is the region's time per launch
    # (inter-launch gaps included, so the roofline fraction is a lower bound)
    per = t0.elapsed_time(t1) / steps
    return per, per, per


def time_decode_graph(torch, pool, synth, m, steps, seed=11):
    """Device time per decode step when `steps` steps are replayed from one CUDA graph (no per-call
    host overhead): the kernel-level number for small m, where launches dominate eager timing.
    Each step takes the next of the pool's disjoint m-slot groups, as in time_decode."""
    groups = slot_groups(torch, pool, synth, m)
    sets = device_inputs(torch, m, steps, seed)
    out = torch.empty((m, HV * D), dtype=torch.bfloat16, device="cuda")
    cap = torch.cuda.Stream()
    s0 = sets[0]
    pool.decode_step(0, groups[0], m, s0["q"], s0["k"], s0["v"], s0["a"], s0["b"], s0["z"], out)  # attributes set
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            for i, s in enumerate(sets):
                ptrs = groups[i % len(groups)]
                pool.decode_step(0, ptrs, m, s["q"], s["k"], s["v"], s["a"], s["b"], s["z"], out, cap)
    graph.replay()  # warm-up
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.current_stream()
    a.record(stream)
    graph.replay()
    b.record(stream)
    torch.cuda.synchronize()
    assert pool.device_status() == 0
    return a.elapsed_time(b) / steps


def time_decode_layers(torch, binding, synth, layers=30, m=M_HEAD, reps=20):
    """One token step of a `layers`-deep stack of GDN layers at m slots (30 x 256 slots, 16 GB of state):
    one decode launch per layer, replayed from a CUDA graph."""
    pool = binding.Pool(HQK, HV, D, D, NUM_SLOTS, layers, W, "bf16", "bf16")
    for layer in range(layers):
        p = synth.layer_params(5, layer, HQK, HV, D, D, W)
        pool.layer_params(layer, *(torch.from_numpy(p[k]) for k in ("conv_w", "A_log", "dt_bias", "norm_w")))
    for _ in range(NUM_SLOTS):
        pool.alloc()
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    for layer in range(layers):
        blk = pool.state_block(layer)
        blk.copy_(torch.randn(blk.shape, generator=g, device="cuda") * math.sqrt(0.1))
    ids = torch.arange(m, dtype=torch.int32, device="cuda")
    ptrs = [pool.slot_ptrs(layer, ids) for layer in range(layers)]
    x = device_inputs(torch, m, 1, 9)[0]
    out = torch.empty((m, HV * D), dtype=torch.bfloat16, device="cuda")
    for layer in range(layers):
        pool.decode_step(layer, ptrs[layer], m, x["q"], x["k"], x["v"], x["a"], x["b"], x["z"], out)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            for layer in range(layers):
                pool.decode_step(layer, ptrs[layer], m, x["q"], x["k"], x["v"], x["a"], x["b"], x["z"], out, cap)
    graph.replay()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.current_stream()
    a.record(stream)
    for _ in range(reps):
        graph.replay()
    b.record(stream)
    torch.cuda.synchronize()
    assert pool.device_status() == 0
    pool.close()
    ms = a.elapsed_time(b) / reps
    return ms


def time_prefill_long(torch, binding, synth, T=80000, reps=3):
    """One 80 000-token prefill (1 250 chunks of 64) into a zeroed slot."""
    pool = binding.Pool(HQK, HV, D, D, 2, 1, W, "bf16", "bf16", max_prefill_tokens=T)
    p = synth.layer_params(5, 0, HQK, HV, D, D, W)
    pool.layer_params(0, *(torch.from_numpy(p[k]) for k in ("conv_w", "A_log", "dt_bias", "norm_w")))
    slot = pool.alloc()
    g = torch.Generator(device="cuda")
    g.manual_seed(80)
    inp = {n: torch.randn((T, w), generator=g, device="cuda").to(torch.bfloat16)
           for n, w in (("q", HQK * D), ("k", HQK * D), ("v", HV * D), ("z", HV * D), ("a", HV), ("b", HV))}
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    ids = torch.tensor([slot], dtype=torch.int32, device="cuda")
    out = torch.empty((T, HV * D), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    times = []
    for r in range(reps + 1):
        pool.recycle(slot, stream)
        pool.alloc()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        pool.prefill_varlen(0, cu, ids, 1, T, inp["q"], inp["k"], inp["v"], inp["a"], inp["b"], inp["z"], out, stream)
        b.record(stream)
        torch.cuda.synchronize()
        if r > 0:
            times.append(a.elapsed_time(b))
    assert pool.device_status() == 0
    pool.close()
    return statistics.median(times)


def time_decode_e2e(torch, pool, synth, m, steps, warmup):
    """Public-API end to end, pipelined the way a serving loop runs it: each step's inputs are copied
    from pinned host memory on a copy-in stream (into one of two device buffer sets) while the
    previous step computes; the decode runs on the compute stream once they have landed; its output
    is copied back to pinned host memory on a copy-out stream while the next step computes.  Events
    order the reuse of both buffer sets.  The timed region runs from before the first input copy to
    after the last output copy, so every step's copies are inside it."""
    ids = torch.tensor(synth.distinct_slots(WORKLOAD_DECODE, m, NUM_SLOTS), dtype=torch.int32, device="cuda")
    ptrs = pool.slot_ptrs(0, ids)
    n_sets = min(steps + warmup, 8)
    host_sets = [{k: v.cpu().pin_memory() for k, v in s.items()} for s in device_inputs(torch, m, n_sets, 7)]
    dev = [{k: torch.empty_like(v, device="cuda") for k, v in host_sets[0].items()} for _ in range(2)]
    out = [torch.empty((m, HV * D), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    out_h = [torch.empty(out[0].shape, dtype=out[0].dtype).pin_memory() for _ in range(2)]
    comp = torch.cuda.current_stream()
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    ev = {n: [torch.cuda.Event() for _ in range(2)] for n in ("in_ready", "in_free", "out_ready", "out_free")}
    for n in ev:  # every event starts out recorded (complete)
        for e in ev[n]:
            e.record(comp)
    h2d = sum(v.numel() * v.element_size() for v in host_sets[0].values())
    d2h = out[0].numel() * out[0].element_size()

    def step(i):
        j = i & 1
        hs = host_sets[i % n_sets]
        cin.wait_event(ev["in_free"][j])  # the decode that read buffer set j (step i - 2) is done
        with torch.cuda.stream(cin):
            for k in dev[j]:
                dev[j][k].copy_(hs[k], non_blocking=True)
        ev["in_ready"][j].record(cin)
        comp.wait_event(ev["in_ready"][j])
        comp.wait_event(ev["out_free"][j])  # step i - 2's output has been copied out
        pool.decode_step(0, ptrs, m, dev[j]["q"], dev[j]["k"], dev[j]["v"], dev[j]["a"], dev[j]["b"], dev[j]["z"],
                         out[j], comp)
        ev["in_free"][j].record(comp)
        ev["out_ready"][j].record(comp)
        cout.wait_event(ev["out_ready"][j])
        with torch.cuda.stream(cout):
            out_h[j].copy_(out[j], non_blocking=True)
        ev["out_free"][j].record(cout)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("e2e_timed")
    t0.record(comp)
    cin.wait_event(t0)
    for i in range(steps):
        step(warmup + i)
    for j in range(2):
        comp.wait_event(ev["out_free"][j])
    t1.record(comp)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    ms = t0.elapsed_time(t1) / steps
    return m / (ms * 1e-3), h2d, d2h


def time_prefill(torch, binding, synth, steps, warmup):
    lengths = PREFILL_LENGTHS
    T = sum(lengths)
    pool = binding.Pool(HQK, HV, D, D, 2 * len(lengths), 1, W, "bf16", "bf16", max_prefill_tokens=T)
    p = synth.layer_params(WORKLOAD_PREFILL, 0, HQK, HV, D, D, W)
    pool.layer_params(0, *(torch.from_numpy(p[k]) for k in ("conv_w", "A_log", "dt_bias", "norm_w")))
    slots = [pool.alloc() for _ in lengths]
    g = torch.Generator(device="cuda")
    g.manual_seed(33)
    inp = {n: torch.randn((T, w), generator=g, device="cuda").to(torch.bfloat16)
           for n, w in (("q", HQK * D), ("k", HQK * D), ("v", HV * D), ("z", HV * D), ("a", HV), ("b", HV))}
    cu = torch.tensor([0] + list(__import__("itertools").accumulate(lengths)), dtype=torch.int32, device="cuda")
    ids = torch.tensor(slots, dtype=torch.int32, device="cuda")
    out = torch.empty((T, HV * D), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()

    def call():
        pool.prefill_varlen(0, cu, ids, len(lengths), T, inp["q"], inp["k"], inp["v"], inp["a"], inp["b"], inp["z"],
                            out, stream)

    for _ in range(warmup):
        for s in slots:
            pool.recycle(s, stream)
            pool.alloc()
        call()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        for s in slots:  # every timed prefill starts from zeroed slots (zeroing is outside the events)
            pool.recycle(s, stream)
            pool.alloc()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda.nvtx.range_push("prefill_timed")
        a.record(stream)
        call()
        b.record(stream)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
        times.append(a.elapsed_time(b))
    assert pool.device_status() == 0
    pool.close()
    return statistics.median(times), T


def time_mixed(torch, binding, synth, iters=5, warmup=2, m=32, lengths=(8192, 8192)):
    """The continuous-batching step of the mixed-batch workload (32 decode slots + two new 8192-token
    prompts per iteration, 16/32 heads, d = 128, bf16 io): gdn_mixed_step against the same work as a
    decode call followed by a prefill call.  Device time per iteration (median); the prompts' slots
    are zeroed outside the timed region, as in a recycled slot."""
    T = sum(lengths)
    pool = binding.Pool(HQK, HV, D, D, m + len(lengths) + 2, 1, W, "bf16", "bf16", max_prefill_tokens=T)
    p = synth.layer_params(WORKLOAD_DECODE, 0, HQK, HV, D, D, W)
    pool.layer_params(0, *(torch.from_numpy(p[k]) for k in ("conv_w", "A_log", "dt_bias", "norm_w")))
    dec = [pool.alloc() for _ in range(m)]
    pre = [pool.alloc() for _ in lengths]
    g = torch.Generator(device="cuda")
    g.manual_seed(44)
    for s in dec:
        pool.state_views(0, s)[0].copy_(torch.randn(pool.state_views(0, s)[0].shape, generator=g, device="cuda") * 0.3)
    d = {n: torch.randn((m, w), generator=g, device="cuda").to(torch.bfloat16)
         for n, w in (("q", HQK * D), ("k", HQK * D), ("v", HV * D), ("z", HV * D), ("a", HV), ("b", HV))}
    x = {n: torch.randn((T, w), generator=g, device="cuda").to(torch.bfloat16)
         for n, w in (("q", HQK * D), ("k", HQK * D), ("v", HV * D), ("z", HV * D), ("a", HV), ("b", HV))}
    ptrs = pool.slot_ptrs(0, torch.tensor(dec, dtype=torch.int32, device="cuda"))
    cu = torch.tensor([0] + list(__import__("itertools").accumulate(lengths)), dtype=torch.int32, device="cuda")
    ids = torch.tensor(pre, dtype=torch.int32, device="cuda")
    dout = torch.empty((m, HV * D), dtype=torch.bfloat16, device="cuda")
    pout = torch.empty((T, HV * D), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()

    def mixed():
        pool.mixed_step(0, ptrs, m, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], dout, cu, ids, len(lengths), T,
                        x["q"], x["k"], x["v"], x["a"], x["b"], x["z"], pout, stream)

    def separate():
        pool.decode_step(0, ptrs, m, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], dout, stream)
        pool.prefill_varlen(0, cu, ids, len(lengths), T, x["q"], x["k"], x["v"], x["a"], x["b"], x["z"], pout, stream)

    def timed(fn):
        times = []
        for it in range(warmup + iters):
            for s in pre:
                pool.recycle(s, stream)
                pool.alloc()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            if it >= warmup:
                times.append(a.elapsed_time(b))
        return statistics.median(times)

    ms_sep = timed(separate)
    ms_mix = timed(mixed)
    assert pool.device_status() == 0
    pool.close()
    return ms_mix, ms_sep, m * decode_bytes_per_slot_step() + prefill_bytes(list(lengths))


def time_proj(torch, binding, reps=20):
    """The layer's projections (16/32 heads, d = 128, hidden 2048, bf16): gdn_in_proj (N = 12 352
    output columns routed to q|k|v|z|a|b) and gdn_out_proj (4096 -> 2048) at the decode batch
    (256 tokens) and the 8-sequence prefill batch (15 998 tokens).  Device time per call (mean over
    `reps` calls replayed from a CUDA graph), with torch.matmul (cuBLAS) on the same product timed
    the same way beside it for context."""
    sh = binding.GdnShape(hqk=HQK, hv=HV, dk=D, dv=D, conv_w=W, chunk=64, io_dtype=1, out_dtype=1, l2_eps=1e-6,
                          norm_eps=1e-6, max_prefill_tokens=0)
    hidden = 2048
    Dq, Dv = HQK * D, HV * D
    N = 2 * Dq + 2 * Dv + 2 * HV
    stream = torch.cuda.current_stream()

    def mean_ms(fn, tag=None):
        """Device time per call: `reps` calls captured in a CUDA graph and replayed, so that the
        host's per-call marshalling (tens of µs from Python) does not pace the small calls."""
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            for _ in range(3):
                fn(cap)
        stream.wait_stream(cap)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            for _ in range(reps):
                fn(cap)
        graph.replay()  # warm replay
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        if tag:
            torch.cuda.nvtx.range_push(tag)
        a.record(stream)
        graph.replay()
        b.record(stream)
        torch.cuda.synchronize()
        if tag:
            torch.cuda.nvtx.range_pop()
        return a.elapsed_time(b) / reps

    out = []
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    w_in = (torch.randn((N, hidden), generator=g, device="cuda") * hidden ** -0.5).to(torch.bfloat16)
    w_out = (torch.randn((hidden, Dv), generator=g, device="cuda") * Dv ** -0.5).to(torch.bfloat16)
    for T in (M_HEAD, sum(PREFILL_LENGTHS)):
        x = torch.randn((T, hidden), generator=g, device="cuda").to(torch.bfloat16)
        o = {n: torch.empty((T, w), dtype=torch.bfloat16, device="cuda")
             for n, w in (("q", Dq), ("k", Dq), ("v", Dv), ("z", Dv), ("a", HV), ("b", HV))}
        y_ref = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
        ms = mean_ms(lambda s: binding.in_proj(sh, hidden, T, x, w_in, o["q"], o["k"], o["v"], o["z"], o["a"],
                                               o["b"], stream=s), tag=f"proj_timed_in_{T}")
        ms_cb = mean_ms(lambda s: torch.matmul(x, w_in.t(), out=y_ref))
        out.append(("in_proj", T, N, hidden, ms, ms_cb))
        ov = torch.randn((T, Dv), generator=g, device="cuda").to(torch.bfloat16)
        y = torch.empty((T, hidden), dtype=torch.bfloat16, device="cuda")
        ms = mean_ms(lambda s: binding.out_proj(sh, hidden, T, ov, w_out, y, stream=s), tag=f"proj_timed_out_{T}")
        ms_cb = mean_ms(lambda s: torch.matmul(ov, w_out.t(), out=y))
        out.append(("out_proj", T, hidden, Dv, ms, ms_cb))
        del x, o, y_ref, ov, y
    return out


def cpu_baseline(seconds=5.0):
    """The fp64 oracle, as it stands, on the host cores, single-thread and on all cores:
    decode at m = 256 (a sample of the 256 slots, all 32 heads; the oracle's cost is linear in the
    slots, so slot-steps/s of the sample is that of the full batch) and prefill tok/s (a prefix of
    the 80 000-token prompt's shape, all 32 heads; linear in tokens)."""
    import numpy as np

    import oracle
    from gated_deltanet_linear_rule_gb300 import synth

    o = oracle.load()
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    p = synth.layer_params(WORKLOAD_DECODE, 0, HQK, HV, D, D, W)
    shape = {"hqk": HQK, "hv": HV, "dk": D, "dv": D, "conv_w": W, "l2_eps": 1e-6, "norm_eps": 1e-6}

    def decode(threads, m_sample):
        slots = synth.distinct_slots(WORKLOAD_DECODE, M_HEAD, NUM_SLOTS)[:m_sample]
        S = np.stack([synth.initial_state(WORKLOAD_DECODE, 0, int(s), HV, D, D) for s in slots]).astype(np.float64)
        conv = np.zeros((m_sample, W - 1, C))
        done, step, el = 0, 0, 0.0
        while el < seconds:
            inp = synth.batch_inputs(WORKLOAD_DECODE, 0, list(range(m_sample)), 1, HQK, HV, D, D, "bf16",
                                     tag="decode", sub=step)
            t0 = time.perf_counter()
            r = o.layer(shape, np.arange(m_sample + 1), inp["q"], inp["k"], inp["v"], inp["a"], inp["b"], inp["z"],
                        p["conv_w"], p["A_log"], p["dt_bias"], p["norm_w"], S, conv, threads=threads)
            el += time.perf_counter() - t0
            S, conv = r["S"], r["convbuf"]
            done += m_sample
            step += 1
        return done / el, f"{step} decode steps of {m_sample} of the 256 slots, all 32 heads, {el:.1f} s"

    def prefill(threads, T):
        inp = synth.token_inputs(5, 0, 0, T, HQK, HV, D, D, "bf16")
        t0 = time.perf_counter()
        o.layer(shape, np.array([0, T]), inp["q"], inp["k"], inp["v"], inp["a"], inp["b"], inp["z"], p["conv_w"],
                p["A_log"], p["dt_bias"], p["norm_w"], np.zeros((1, HV, D, D)), np.zeros((1, W - 1, C)),
                threads=threads)
        el = time.perf_counter() - t0
        return T / el, f"the first {T} tokens of an 80 000-token prompt (one sequence, all 32 heads), {el:.1f} s"

    dec_all, dec_all_s = decode(cores, 16)
    dec_one, dec_one_s = decode(1, 2)
    pre_all, pre_all_s = prefill(cores, 8192)
    pre_one, pre_one_s = prefill(1, 2048)
    return {"value": dec_all, "unit": UNIT, "cores": cores, "threads": cores, "kind": "oracle",
            "sample": dec_all_s,
            "decode_single_thread": {"value": dec_one, "unit": UNIT, "threads": 1, "sample": dec_one_s},
            "prefill": {"value": pre_all, "unit": "tok/s", "threads": cores, "sample": pre_all_s},
            "prefill_single_thread": {"value": pre_one, "unit": "tok/s", "threads": 1, "sample": pre_one_s}}


def run_ours(args):
    import torch

    from gated_deltanet_linear_rule_gb300 import binding, synth

    rank, world, local = dist_init()
    torch.cuda.set_device(local)
    hbm, bf16, peak_kind = peaks()
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(local).uuid)
        uuid = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
    except Exception:
        uuid = None

    pool = make_decode_pool(torch, binding, synth)
    barrier(world)
    clocks = ClockSampler(uuid)
    clocks.start()
    torch.cuda.synchronize()
    barrier(world)
    wall0 = time.perf_counter()
    step_ms, kern_mean, kern_med = time_decode(torch, pool, synth, M_HEAD, args.steps, args.warmup)
    wall = time.perf_counter() - wall0
    ck = clocks.stop()
    step_ms = reduce_max(step_ms, world)
    value = world * M_HEAD / (step_ms * 1e-3)

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": HEAD_WORKLOAD, "m": M_HEAD, "pool_slots": NUM_SLOTS, "io": "bf16",
                   "state": "fp32 N(0,0.1)", "parallelism": f"replicas x{world}",
                   "l2": f"no flush: inputs larger than L2 ({M_HEAD * HV * D * D * 4 / 1e6:.0f} MB of state per step)"},
        "gpu_launches": args.steps,
    }
    algo = M_HEAD * decode_bytes_per_slot_step() + decode_param_bytes()
    ach = algo / (kern_mean * 1e-3) / 1e9
    result["roofline"] = {"kernel": "decode_kernel<128,bf16,bf16,4>", "bound": "hbm", "achieved": ach, "peak": hbm,
                          "unit": "GB/s", "frac": ach / hbm, "peak_kind": peak_kind,
                          "frac_of_8TBs": ach / 8000.0,
                          "traffic": profiled_traffic("decode_kernel<128,bf16,bf16,4>", DECODE_SOURCES, M_HEAD),
                          "bytes_per_launch": algo, "launch_ms": kern_mean,
                          "launch_ms_method": "timed region / launches, back to back (inter-launch gaps included)"}
    if ck:
        result["clocks"] = {"sm_mhz": ck["sm_mhz"], "sm_max_mhz": ck["sm_max_mhz"], "reasons": ck["reasons"],
                            "samples": ck["samples"]}
    if rank == 0 and not args.no_sweep:
        sweep = []
        for m in SWEEP:
            sm, km, _ = time_decode(torch, pool, synth, m, max(10, min(args.steps, 500)), 3, seed=100 + m)
            gm = time_decode_graph(torch, pool, synth, m, 100, seed=200 + m)
            b = m * decode_bytes_per_slot_step() + decode_param_bytes()
            sweep.append({"m": m, "bytes_per_step": b, "slot_steps_per_s": m / (sm * 1e-3), "us_per_step": sm * 1e3,
                          "gbs": b / (km * 1e-3) / 1e9, "frac": b / (km * 1e-3) / 1e9 / hbm,
                          "graph_us_per_step": gm * 1e3, "graph_slot_steps_per_s": m / (gm * 1e-3),
                          "graph_frac": b / (gm * 1e-3) / 1e9 / hbm})
        result["decode_sweep"] = {
            "method": "each step on the next of the 256-slot pool's disjoint m-slot groups (so a step's states "
                      "were last touched 256/m - 1 steps earlier, with more than the 129 MB L2 of other states in "
                      "between: HBM, not L2); eager: back-to-back launches; graph: 100 steps replayed from one "
                      "CUDA graph",
            "points": sweep}
    if rank == 0:
        e2e, h2d, d2h = time_decode_e2e(torch, pool, synth, M_HEAD, min(args.steps, 2000), args.warmup)
        result["e2e"] = {"value": e2e * world, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                         "method": "pinned host inputs copied in on a copy-in stream and each step's output copied "
                                   "back on a copy-out stream, overlapping the neighbouring steps' kernels; every "
                                   "step's copies inside the timed region, which has no per-step event records "
                                   "(the device-timed loop records two per step)"}
    pool.close()
    if rank == 0 and not args.no_prefill:
        pms, T = time_prefill(torch, binding, synth, max(3, min(args.steps, 10)), 2)
        pb = prefill_bytes(PREFILL_LENGTHS)
        flops = PREFILL_FLOPS_PER_TOKEN * T
        traffic = profiled_traffic("chunked_prefill_varlen8", PREFILL_SOURCES, 1)
        result["prefill"] = {"workload": "8 sequences {1,17,300,4095,1024,2048,513,8000}, bf16 io, zero state",
                             "tokens": T, "ms": pms, "tok_per_s": T / (pms * 1e-3),
                             "gbs": pb / (pms * 1e-3) / 1e9, "frac_hbm": pb / (pms * 1e-3) / 1e9 / hbm,
                             "bytes": pb, "tflops": flops / (pms * 1e-3) / 1e12,
                             "frac_tensor": flops / (pms * 1e-3) / 1e12 / bf16,
                             "bound": "hbm (137 flop/B < ridge 279)",
                             # DRAM bytes the two passes move (ncu, this source): the records between them
                             "traffic": traffic,
                             "traffic_gbs": traffic / (pms * 1e-3) / 1e9 if traffic else None}
        lms = time_prefill_long(torch, binding, synth)
        result["prefill_80k"] = {"workload": "one 80 000-token prefill, bf16 io, zero state", "ms": lms,
                                 "tok_per_s": 80000 / (lms * 1e-3),
                                 "frac_hbm": prefill_bytes([80000]) / (lms * 1e-3) / 1e9 / hbm}
        mix, sep, mb = time_mixed(torch, binding, synth)
        result["mixed_step"] = {"workload": "gdn_mixed_step: 32 decode slots + two 8192-token prompts into zeroed "
                                            "slots, bf16 io (the mixed-batch iteration)",
                                "ms": mix, "ms_separate_calls": sep, "bytes": mb,
                                "gbs": mb / (mix * 1e-3) / 1e9, "frac_hbm": mb / (mix * 1e-3) / 1e9 / hbm}
        l30 = time_decode_layers(torch, binding, synth)
        result["decode_30_layers"] = {"workload": "one token step of 30 stacked GDN layers at m = 256 "
                                                  "(30 x 256 slots, 16.1 GB of state), CUDA-graph replay",
                                      "ms_per_token_step": l30, "tokens_per_s": M_HEAD / (l30 * 1e-3),
                                      "slot_steps_per_s": 30 * M_HEAD / (l30 * 1e-3)}
    if rank == 0 and not args.no_proj:
        proj = []
        for name, T, N, K, ms, ms_cb in time_proj(torch, binding):
            tf = 2.0 * T * N * K / (ms * 1e-3) / 1e12
            proj.append({"call": name, "tokens": T, "n": N, "k": K, "us": ms * 1e3, "tflops": tf,
                         "frac_tensor": tf / bf16, "cublas_us": ms_cb * 1e3})
        result["projections"] = {"workload": "gdn_in_proj (2048 -> 12 352 columns: q|k|v|z|a|b) and gdn_out_proj "
                                             "(4096 -> 2048), bf16, at the decode batch and the 8-sequence "
                                             "prefill batch; cuBLAS (torch.matmul) on the same product beside it",
                                 "bound": "tensor", "peak_tflops": bf16, "calls": proj}
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    result["wall_s_timed_region"] = wall
    if rank == 0:
        print(json.dumps(result))
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def run_reference(args):
    """The fp64 CPU oracle, as it stands, on the host cores: same metric, bounded sample per step."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import numpy as np

    import oracle
    from gated_deltanet_linear_rule_gb300 import synth

    o = oracle.load()
    p = synth.layer_params(WORKLOAD_DECODE, 0, HQK, HV, D, D, W)
    shape = {"hqk": HQK, "hv": HV, "dk": D, "dv": D, "conv_w": W, "l2_eps": 1e-6, "norm_eps": 1e-6}
    m_sample = 8
    slots = synth.distinct_slots(WORKLOAD_DECODE, M_HEAD, NUM_SLOTS)[:m_sample]
    S = np.stack([synth.initial_state(WORKLOAD_DECODE, 0, int(s), HV, D, D) for s in slots]).astype(np.float64)
    conv = np.zeros((m_sample, W - 1, C))
    times = []
    for step in range(args.warmup + args.steps):
        inp = synth.batch_inputs(WORKLOAD_DECODE, 0, list(range(m_sample)), 1, HQK, HV, D, D, "bf16",
                                 tag="decode", sub=step)
        t0 = time.perf_counter()
        r = o.layer(shape, np.arange(m_sample + 1), inp["q"], inp["k"], inp["v"], inp["a"], inp["b"], inp["z"],
                    p["conv_w"], p["A_log"], p["dt_bias"], p["norm_w"], S, conv)
        el = time.perf_counter() - t0
        S, conv = r["S"], r["convbuf"]
        if step >= args.warmup:
            times.append(el)
    ms = 1e3 * sum(times) / len(times)
    value = m_sample / (ms * 1e-3)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": HEAD_WORKLOAD, "m": M_HEAD, "pool_slots": NUM_SLOTS, "io": "bf16",
                   "parallelism": "host cores (OpenMP over slot x head)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": o.max_threads(), "kind": "oracle",
                         "sample": f"each step: {m_sample} of the 256 slots, all 32 heads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def run_profile_case(args):
    """One small case only, for an ncu capture of its kernels: `decode256` (the m = 256 decode on the
    256-slot pool, 0.54 GB of state) or `prefill8` (the 8-sequence, 15 998-token prefill, under 2 GB
    with its workspace): W warm-up launches (calls), then K.  Prints one line naming the case and its
    time; it is not a bench line."""
    import torch

    from gated_deltanet_linear_rule_gb300 import binding, synth

    torch.cuda.set_device(0)
    if args.profile_case == "decode256":
        pool = make_decode_pool(torch, binding, synth)
        ms, _, _ = time_decode(torch, pool, synth, M_HEAD, args.steps, args.warmup)
        pool.close()
    else:
        ms, _ = time_prefill(torch, binding, synth, args.steps, args.warmup)
    print(json.dumps({"profile_case": args.profile_case, "warmup": args.warmup, "steps": args.steps,
                      "ms_per_call": ms}))


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1, help="ranks (one per GPU, launched by torchrun for N > 1)")
    ap.add_argument("--steps", type=int, default=5000, help="timed decode steps at m = 256")
    ap.add_argument("--warmup", type=int, default=5, help="untimed warm-up steps (at least 3 are run)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"],
                    help="ours: the CUDA library; reference: the fp64 oracle on the host cores")
    ap.add_argument("--no-sweep", action="store_true", help="skip the m-sweep and graph-replay timings")
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip the prefill, 80k prefill, mixed-step and 30-layer timings")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle baseline sample")
    ap.add_argument("--no-proj", action="store_true", help="skip the in_proj / out_proj timings")
    ap.add_argument("--cpu-seconds", type=float, default=5.0,
                    help="length of each decode sample of the oracle baseline (single-thread and all cores)")
    ap.add_argument("--profile-case", choices=["decode256", "prefill8"], default=None,
                    help="run only this small case (for an ncu capture of its kernels) and print its time")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)  # at least 3 untimed warm-up steps, whatever was asked
    if args.profile_case:
        run_profile_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
