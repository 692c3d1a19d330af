#!/usr/bin/env python
"""Decode MoE expert block on GB300: throughput of the full layer stack, one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--tokens M]
    python bench.py --impl reference ...        # the fp64 CPU oracle on the host cores

A step is one decode step through every layer of the stack (both phases of every layer in one
persistent cooperative kernel launch, replayed as a CUDA graph), on seeded synthetic weights drawn
in HBM and token inputs already resident on the device.  Each step uses the next of several
pre-drawn input sets, so expert ids change from step to step, and a step reads far more weight
bytes than L2 holds.

value      tokens per second through the whole stack (all ranks), timed with CUDA events
e2e        the same through moe_stack_step_host: inputs copied from pinned host memory and the
           output copied back inside the timed region
roofline   the fused stack kernel (the only kernel of a step): algorithmic bytes of one step
           divided by the step's device time
separate_kernels  the same layers through the two-kernel mode (kernel A then kernel B per layer),
           each phase replayed alone: per-launch bytes and time, for comparison
cpu_baseline  the oracle, as it stands, on a bounded sample of the same workload
N > 1      independent replicas, one per GPU (the block has no exchange step); weak scaling
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from quantized_moe_expert_dequant_gb300 import synth  # noqa: E402
from quantized_moe_expert_dequant_gb300.workloads import ALL, Shape  # noqa: E402

METRIC = "MoE decode tok/s (full layer stack) and achieved HBM GB/s vs peak, 1 GB300"
DEFAULT_WORKLOAD = "qwen3_stack_8bit"
NORM_EPS = 1e-6   # RMSNorm epsilon of the chained stack (--chain-norm)
GEMV_NAMES = ("qwen25_1p5b_qo", "qwen25_1p5b_kv", "qwen3_8b_qo", "qwen3_8b_kv")
KERNEL_SOURCES = ["quantized_moe_expert_dequant_gb300/csrc/moe_cols.cuh",
                  "quantized_moe_expert_dequant_gb300/csrc/moe_cols_g8.cu",
                  "quantized_moe_expert_dequant_gb300/csrc/moe_kernels.cu",
                  "quantized_moe_expert_dequant_gb300/csrc/moe_fused.cuh",
                  "quantized_moe_expert_dequant_gb300/csrc/moe_kernels_g8.cu",
                  "quantized_moe_expert_dequant_gb300/csrc/moe_grouped.cuh",
                  "quantized_moe_expert_dequant_gb300/csrc/moe_kernels.cuh",
                  "quantized_moe_expert_dequant_gb300/csrc/moe_phases.cuh",
                  "quantized_moe_expert_dequant_gb300/csrc/moe_tma.cuh",
                  "quantized_moe_expert_dequant_gb300/csrc/moe_common.cuh",
                  "quantized_moe_expert_dequant_gb300/csrc/moe_timeline.cuh"]


# ---------------------------------------------------------------- algorithmic bytes

def proj_bytes(rows, cols, bits):
    return rows * cols * bits // 8 + (rows * cols // 64) * 4


def layer_bytes(shape: Shape, m: int, unique_experts: int, first_layer: bool,
                chained: bool = False):
    """(kernel A bytes, kernel B bytes) of one layer for m tokens whose slots name
    `unique_experts` distinct experts: each selected weight byte is counted once.  A chained
    layer after the first reads the previous output (fp32) and the norm weight instead of x."""
    act = shape.top_k * shape.dff + shape.n_shared * shape.dff_shared
    a = unique_experts * (proj_bytes(shape.dff, shape.din, shape.bits_gate)
                          + proj_bytes(shape.dff, shape.din, shape.bits_up))
    a += shape.n_shared * 2 * proj_bytes(shape.dff_shared, shape.din, shape.bits_shared)
    normed = chained and not first_layer
    a += m * ((shape.din * 4 if normed else shape.din * 2) + act * 4 + shape.top_k * 8)
    if normed:
        a += shape.din * 2
    if shape.n_shared and shape.shared_gate:
        a += shape.din * 2
    b = unique_experts * proj_bytes(shape.din, shape.dff, shape.bits_down)
    b += shape.n_shared * proj_bytes(shape.din, shape.dff_shared, shape.bits_shared)
    b += m * (act * 4 + shape.din * (2 if first_layer else 4) + shape.din * 4 + shape.top_k * 4)
    return a, b


# ---------------------------------------------------------------- inputs

def input_set(shape: Shape, m: int, step: int, chained: bool = False):
    L = shape.layers
    x = np.stack([np.stack([synth.activations(shape.seed, l, t + 1000 * step, shape.din)
                            for t in range(m)]) for l in range(1 if chained else L)])
    ids = np.stack([np.stack([synth.topk_ids(shape.seed, l, t, shape.n_experts, shape.top_k, step)
                              for t in range(m)]) for l in range(L)]).astype(np.int32)
    sc = np.stack([np.stack([synth.scores(shape.seed, l, t, shape.top_k, step)
                             for t in range(m)]) for l in range(L)]).astype(np.float32)
    resid0 = np.stack([synth.residual(shape.seed, 0, t + 1000 * step, shape.din) for t in range(m)])
    return x, ids.reshape(L, m, shape.top_k), sc.reshape(L, m, shape.top_k), resid0


def unique_per_layer(ids: np.ndarray):
    return [len(set(ids[l].reshape(-1).tolist())) for l in range(ids.shape[0])]


# ---------------------------------------------------------------- the oracle on the host

def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_layer_calls(shape: Shape, layers):
    """One call per layer: that layer's block term (every output row, every slot and shared
    expert, residual zero) for token 0 of input set 0 through the unchanged oracle_moe_token.  A
    layer's block term depends only on its own seeded inputs, so layers are independent units of
    work.  The packed experts are drawn on the host here, outside any timing."""
    from oracle import oracle as O
    x, ids, sc, _ = input_set(shape, 1, 0)
    zero = np.zeros(shape.din, np.float32)
    calls = []
    for l in layers:
        pk = lambda proj, e, r, c, b, l=l: O.Packed(*synth.expert_proj(shape.seed, l, proj, e, r, c, b), b)
        slots = [int(e) for e in ids[l][0]]
        kw = dict(scores=sc[l][0],
                  gate=[pk(synth.GATE, e, shape.dff, shape.din, shape.bits_gate) for e in slots],
                  up=[pk(synth.UP, e, shape.dff, shape.din, shape.bits_up) for e in slots],
                  down=[pk(synth.DOWN, e, shape.din, shape.dff, shape.bits_down) for e in slots])
        if shape.n_shared:
            w, b = shape.dff_shared, shape.bits_shared
            kw.update(sh_gate=[pk(synth.SH_GATE, t, w, shape.din, b) for t in range(shape.n_shared)],
                      sh_up=[pk(synth.SH_UP, t, w, shape.din, b) for t in range(shape.n_shared)],
                      sh_down=[pk(synth.SH_DOWN, t, shape.din, w, b) for t in range(shape.n_shared)],
                      gate_vec_bf16=synth.gate_vector(shape.seed, l, shape.din)
                      if shape.shared_gate else None)
        calls.append(lambda kw=kw, xl=x[l][0]: O.moe_token(xl, zero, **kw))
    return calls


class OracleStack:
    """The oracle on every host core: one step is every layer of the stack, one layer per thread
    at a time (ctypes releases the GIL inside the oracle), so a step's wall time is measured,
    not extrapolated."""

    def __init__(self, shape: Shape, cores: int):
        import concurrent.futures as cf
        self.shape, self.cores = shape, cores
        self.calls = oracle_layer_calls(shape, range(shape.layers))
        self.pool = cf.ThreadPoolExecutor(max_workers=cores)

    def step(self) -> float:
        t0 = time.perf_counter()
        list(self.pool.map(lambda c: c(), self.calls))
        return time.perf_counter() - t0

    def close(self):
        self.pool.shutdown()


def oracle_baseline(shape: Shape, steps: int = 3) -> dict:
    """Median of `steps` timed steps of the whole stack (one token) on all host cores."""
    cores = host_cores()
    os_ = OracleStack(shape, cores)
    os_.step()                                            # warm-up (page-in, thread start)
    times = [os_.step() for _ in range(steps)]
    os_.close()
    t = statistics.median(times)
    layers_s = shape.layers / t
    return {"value": 1.0 / t, "unit": "tok/s", "cores": cores, "kind": "oracle",
            "layers_per_s": layers_s, "gbs": layers_s * per_token_layer_weight_bytes(shape) / 1e9,
            "sample": f"median of {steps} steps of the whole {shape.layers}-layer stack (every "
                      f"output row, every slot, one token) through the unchanged fp64 oracle, "
                      f"one layer per thread on {cores} host cores ({t:.2f} s per step)"}


def per_token_layer_weight_bytes(shape: Shape):
    return shape.top_k * shape.expert_bytes() + shape.shared_bytes()


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi every 100 ms from construction to stop(); stop(t0, t1) keeps the samples taken
    between two wall-clock datetimes (the timed region) when there are any."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.proc = None
        try:
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "100"]
            if bus_id:
                cmd += ["-i", bus_id]
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None

    def stop(self, t0=None, t1=None):
        import datetime as dt
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.strip().splitlines():
            r = line.split(", ")
            if len(r) < 10:
                continue
            try:
                when = dt.datetime.strptime(r[0].strip(), "%Y/%m/%d %H:%M:%S.%f")
            except ValueError:
                when = None
            rows.append((when, r[1:]))
        window = False
        if t0 is not None and t1 is not None:
            inside = [x for x in rows if x[0] is not None and t0 <= x[0] <= t1]
            if inside:
                rows, window = inside, True
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "timed_region_only": window}


# ---------------------------------------------------------------- helpers

def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return None


def code_only(text: str) -> str:
    """C/C++/CUDA source without comments and with runs of whitespace collapsed, so that the
    hash below changes with the code, not with its comments."""
    import re
    out, i, n = [], 0, len(text)
    while i < n:
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif text[i] in "\"'":
            q, j = text[i], i + 1
            while j < n and text[j] != q:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(text[i])
            i += 1
    return re.sub(r"\s+", " ", "".join(out)).strip()


def kernel_source_hash() -> str:
    """Hash of the dominant kernels' code (comments and layout ignored): a DRAM-traffic record
    in profiles/traffic.txt is used only while it matches."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(code_only(open(os.path.join(ROOT, f), encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str, layers: int):
    """dram bytes per launch of `layers` layers from the committed ncu summary, if taken on the
    current source: the record's bytes per launch of its own layer count, scaled by the layers
    (the kernel's traffic is per layer)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    src = kernel_source_hash()
    for line in open(path):
        kv = dict(p.split("=", 1) for p in line.split() if "=" in p)
        if kv.get("kernel") == kernel and kv.get("workload") == workload and kv.get("src") == src:
            per = float(kv["dram_bytes_per_launch"])
            rec_layers = int(kv.get("layers", layers))
            return per * layers / rec_layers
    return None


def dist_setup(backend):
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return rank, world, local


def max_over_ranks(v: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, ms_local: float, device=None):
    """Whole-job rate: the units every rank processed over the slowest rank's time.
    Returns (units per second, the max-over-ranks milliseconds)."""
    import torch.distributed as dist
    world = dist.get_world_size() if dist.is_available() and dist.is_initialized() else 1
    ms = max_over_ranks(ms_local, device)
    return world * units_per_rank / (ms / 1e3), ms


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------- the reference arm

def run_reference(args, shape: Shape):
    rank, world, _ = dist_setup("gloo")
    if rank != 0:
        return 0
    # each step: every layer of the stack through the oracle, on every host core
    cores = host_cores()
    os_ = OracleStack(shape, cores)
    for _ in range(args.warmup):
        os_.step()
    times = [os_.step() for _ in range(args.steps)]
    os_.close()
    spent = sum(times)
    tok = args.steps / spent
    layers_s = shape.layers * tok
    line = {
        "impl": "reference", "metric": METRIC, "value": tok, "unit": "tok/s", "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": spent / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": shape.name, "layers": shape.layers, "tokens_per_step": 1},
        "cpu_baseline": {"value": tok, "unit": "tok/s", "cores": cores, "kind": "oracle",
                         "layers_per_s": layers_s,
                         "sample": f"each step the whole {shape.layers}-layer stack (every "
                                   f"output row, every slot, one token) through the unchanged "
                                   f"fp64 oracle, one layer per thread on {cores} host cores; "
                                   f"{args.steps} steps in {spent:.1f} s"},
        "e2e": {"value": tok, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm

def mode_of(kernels: str) -> int:
    from quantized_moe_expert_dequant_gb300 import binding as Bn
    return {"fused": Bn.KERNELS_FUSED, "separate": Bn.KERNELS_SEPARATE,
            "columns": Bn.KERNELS_COLUMNS, "columns-ahead": Bn.KERNELS_COLUMNS_AHEAD,
            "mma": Bn.KERNELS_MMA, "pool": Bn.KERNELS_POOL}[kernels]


def run_ours(args, shape: Shape):
    import torch

    from quantized_moe_expert_dequant_gb300 import binding as Bn

    rank, world, local = dist_setup("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    m, L, S = args.tokens, shape.layers, args.input_sets

    bus = None
    try:
        bus = torch.cuda.get_device_properties(device).pci_bus_id
    except AttributeError:
        bus = None
    sampler = ClockSampler(bus if bus else str(local))   # running long before the timed region

    free, _ = torch.cuda.mem_get_info()
    need = shape.layer_weight_bytes() * L
    if free < need * 1.05:
        raise SystemExit(f"workload needs {need / 1e9:.1f} GB, {free / 1e9:.1f} GB free")
    layers = [Bn.synth_layer_device(shape, l) for l in range(L)]
    chained = args.chain_norm
    kernels = args.kernels
    if kernels == "auto":   # one token: the column split; a batch: the tensor-core tiles
        cols_ok = (m == 1 and not chained and shape.bits_gate in (4, 8) and shape.din <= 4096)
        mma_ok = (m > 1 and not chained and m <= 64 and m * shape.top_k <= 256
                  and shape.n_experts <= 1024)
        kernels = "columns" if cols_ok else "mma" if mma_ok else "fused"
    mode = mode_of(kernels)
    norm = None
    if chained and L > 1:
        rows = np.stack([synth.norm_weight(shape.seed, l, shape.din) for l in range(1, L)])
        norm = torch.from_numpy(rows.view(np.int16)).view(torch.bfloat16).to(device)
    elif chained:
        norm = torch.ones((1, shape.din), dtype=torch.bfloat16, device=device)
    stack = Bn.MoeStack(layers, max_tokens=m, kernel_mode=mode, norm_weight=norm, eps=NORM_EPS)
    parts_stack = Bn.MoeStack(layers, max_tokens=m, kernel_mode=Bn.KERNELS_SEPARATE,
                              norm_weight=norm, eps=NORM_EPS)

    def dev(a, dt):
        a = np.ascontiguousarray(a)
        if dt == torch.bfloat16:
            return torch.from_numpy(a.view(np.int16)).view(dt).to(device)
        return torch.from_numpy(a).to(device)

    sets, uniq = [], []
    for s in range(S):
        x, ids, sc, r0 = input_set(shape, m, s, chained)
        uniq.append(unique_per_layer(ids))
        sets.append((dev(x, torch.bfloat16), dev(ids, torch.int32), dev(sc, torch.float32),
                     dev(r0, torch.bfloat16), torch.empty((m, shape.din), dtype=torch.float32,
                                                          device=device), (x, ids, sc, r0)))
    bytes_a = [sum(layer_bytes(shape, m, u[l], l == 0, chained)[0] for l in range(L))
               for u in uniq]
    bytes_b = [sum(layer_bytes(shape, m, u[l], l == 0, chained)[1] for l in range(L))
               for u in uniq]

    stream = torch.cuda.current_stream(device)
    ab_stack, ab_kernels = None, None
    if args.ab:
        ab_kernels = args.ab
        ab_stack = Bn.MoeStack(layers, max_tokens=m, kernel_mode=mode_of(ab_kernels),
                               norm_weight=norm, eps=NORM_EPS)

    def step(i, parts=3, st=None):
        x, ids, sc, r0, out, _ = sets[i % S]
        if parts == 3:
            (st or stack).step(x, ids, sc, r0, out, stream)
        else:
            parts_stack.step_parts(parts, x, ids, sc, r0, out, stream)

    def time_steps(n_steps, st=None):
        """ms per step of n_steps replays, CUDA events on the launching stream."""
        torch.cuda.synchronize(device)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for i in range(n_steps):
            step(i, st=st)
        a1.record(stream)
        torch.cuda.synchronize(device)
        return a0.elapsed_time(a1) / n_steps

    # warm-up: captures every graph, then W untimed steps
    for i in range(S):
        step(i)
        step(i, Bn.PART_GATE_UP)
        step(i, Bn.PART_DOWN)
        if ab_stack is not None:
            step(i, st=ab_stack)
    torch.cuda.synchronize(device)
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(device)
    assert stack.get_error() == 0

    # timed region: exactly K steps
    import datetime as dt
    tw0 = dt.datetime.now()
    barrier(device)
    torch.cuda.synchronize(device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize(device)
    barrier(device)
    ms_local = e0.elapsed_time(e1)
    value, ms = job_rate(m * args.steps, ms_local, device)
    ms_per_step = ms / args.steps

    # the sampling protocol, after the K steps: >= 10 samples of >= 5 replays (about 100 ms each,
    # so the clock sampler sees them); with --ab the other kernel mode's samples alternate with
    # this one's
    reps = max(5, int(np.ceil(100.0 / max(ms_per_step, 1e-3))))
    samp_a, samp_b = [], []
    for _ in range(max(10, args.samples)):
        samp_a.append(time_steps(reps))
        if ab_stack is not None:
            samp_b.append(time_steps(reps, ab_stack))
    tw1 = dt.datetime.now()

    def sample_stats(v):
        v = np.asarray(v)
        med = float(np.median(v))
        return {"n": len(v), "replays": reps, "ms_per_step_median": med,
                "ms_per_step_min": float(v.min()), "ms_per_step_max": float(v.max()),
                "spread": float((v.max() - v.min()) / med),
                "value_median": world * m / (med * 1e-3) * (L if args.single_layer else 1)}
    step_bytes = sum(bytes_a[i % S] + bytes_b[i % S] for i in range(args.steps)) / args.steps

    # the two-kernel mode, each phase of every layer replayed alone (for comparison)
    reps = max(args.steps // 4, 20)

    def time_part(parts):
        torch.cuda.synchronize(device)
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for i in range(reps):
            step(i, parts)
        a1.record(stream)
        torch.cuda.synchronize(device)
        return a0.elapsed_time(a1) / (reps * L * m)   # ms per launch

    ms_a = time_part(Bn.PART_GATE_UP)
    ms_b = time_part(Bn.PART_DOWN)
    mean_a = sum(bytes_a[i % S] for i in range(reps)) / reps / (L * m)
    mean_b = sum(bytes_b[i % S] for i in range(reps)) / reps / (L * m)

    # end to end through the public host-buffer call
    pinned = []
    for (_, _, _, _, _, host) in sets:
        x, ids, sc, r0 = host
        pin = lambda a, dt: (torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(dt)
                             if dt == torch.bfloat16 else torch.from_numpy(np.ascontiguousarray(a))
                             ).pin_memory()
        pinned.append((pin(x, torch.bfloat16), pin(ids, torch.int32), pin(sc, torch.float32),
                       pin(r0, torch.bfloat16),
                       torch.empty((m, shape.din), dtype=torch.float32).pin_memory()))
    for i in range(min(3, len(pinned))):
        stack.step_host(*pinned[i], stream=stream)
    e2e_steps = max(args.steps // 4, 10)
    barrier(device)
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        stack.step_host(*pinned[i % S], stream=stream)
    t1 = time.perf_counter()
    barrier(device)
    e2e_s = max_over_ranks(t1 - t0, device)
    h2d = sum(t.numel() * t.element_size() for t in pinned[0][:4])
    d2h = pinned[0][4].numel() * 4
    clocks = sampler.stop(tw0, tw1)
    assert stack.get_error() == 0 and parts_stack.get_error() == 0
    assert ab_stack is None or ab_stack.get_error() == 0

    peaks = measured_peaks()
    peak = peaks["hbm_gbs"] if peaks else 6800.0
    peak_note = "of measured" if peaks else "of fallback"
    ach_a = mean_a / (ms_a * 1e-3) / 1e9
    ach_b = mean_b / (ms_b * 1e-3) / 1e9
    one_launch = (Bn.KERNELS_FUSED, Bn.KERNELS_COLUMNS, Bn.KERNELS_COLUMNS_AHEAD,
                  Bn.KERNELS_POOL)
    dominant = {Bn.KERNELS_FUSED: "fused_kernel", Bn.KERNELS_POOL: "fused_kernel",
                Bn.KERNELS_COLUMNS: "cols_kernel",
                Bn.KERNELS_COLUMNS_AHEAD: "cols_kernel",
                Bn.KERNELS_MMA: "mma path (route, gate_up_mma, down_mma, tail per layer)"
                }.get(mode, "gate_up_kernel")
    if mode in one_launch or mode == Bn.KERNELS_MMA:
        # the step's bytes over the step's device time (one launch per step, or the tensor-core
        # path's four launches per layer taken together)
        ach, per_launch_bytes, per_launch_us = (step_bytes / (ms_per_step * 1e-3) / 1e9,
                                                step_bytes, ms_per_step * 1e3)
    else:
        ach, per_launch_bytes, per_launch_us = ach_a, mean_a, ms_a * 1e3
    traffic = (None if mode == Bn.KERNELS_COLUMNS_AHEAD else
               profiled_traffic(dominant, args.workload + ("_chained" if chained else ""), L))

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_baseline(shape)
        if args.single_layer:
            cpu["value"], cpu["unit"] = cpu["layers_per_s"], "layers/s"

    unit = "tok/s"
    if args.single_layer:   # one layer per replica: layers per second (SURVEY units)
        value *= L
        unit = "layers/s"
    line = {
        "metric": METRIC, "value": value, "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded weights drawn in HBM, seeded token inputs)",
        "config": {"workload": shape.name, "din": shape.din, "dff": shape.dff,
                   "experts": shape.n_experts, "top_k": shape.top_k,
                   "bits": [shape.bits_gate, shape.bits_up, shape.bits_down],
                   "shared": [shape.n_shared, shape.dff_shared, shape.bits_shared],
                   "layers": L, "tokens_per_step": m, "input_sets": S,
                   "chain_norm": bool(chained), "kernels": kernels,
                   "ids_known_ahead": mode == Bn.KERNELS_COLUMNS_AHEAD,
                   "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: {step_bytes / 1e9:.3f} GB of selected weights "
                         f"per step, ids re-drawn per step"},
        "hbm": {"step_bytes": step_bytes, "step_gbs": step_bytes / (ms_per_step * 1e-3) / 1e9,
                "peak_gbs": peak, "frac": step_bytes / (ms_per_step * 1e-3) / 1e9 / peak,
                "note": peak_note},
        "roofline": {"kernel": dominant, "bound": "hbm", "achieved": ach, "peak": peak,
                     "unit": "GB/s", "frac": ach / peak, "traffic": traffic,
                     # far above the copy peak means the timed kernel skipped bytes
                     "sanity": ("ok" if ach <= 1.1 * peak else
                                "achieved bandwidth above 1.1x the copy peak: harness error"),
                     "bytes_per_launch": per_launch_bytes, "us_per_launch": per_launch_us,
                     "note": peak_note + " (copy peak)"},
        "separate_kernels": {
            "gate_up_kernel": {"achieved": ach_a, "frac": ach_a / peak,
                               "bytes_per_launch": mean_a, "us_per_launch": ms_a * 1e3},
            "down_kernel": {"achieved": ach_b, "frac": ach_b / peak,
                            "bytes_per_launch": mean_b, "us_per_launch": ms_b * 1e3}},
        "cpu_baseline": cpu,
        "e2e": {"value": world * m * e2e_steps / e2e_s * (L if args.single_layer else 1),
                "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": (args.steps if mode in one_launch else
                         args.steps * L * 4 if mode == Bn.KERNELS_MMA else args.steps * L * m * 2),
        "clocks": clocks,
        "samples": sample_stats(samp_a),
    }
    if args.single_layer:
        line["config"]["replicas"] = L
        if shape.din == 2048 and shape.dff == 768 and shape.top_k == 8:
            line["tok_equivalent_48_layers"] = value / 48
    if ab_stack is not None:
        sa, sb = sample_stats(samp_a), sample_stats(samp_b)
        line["ab"] = {"kernels": [kernels, ab_kernels], "alternated_samples": len(samp_a),
                      "ms_per_step_median": [sa["ms_per_step_median"], sb["ms_per_step_median"]],
                      "spread": [sa["spread"], sb["spread"]],
                      "b_over_a_time": sb["ms_per_step_median"] / sa["ms_per_step_median"]}
        ab_stack.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    stack.close()
    parts_stack.close()
    return 0


# ---------------------------------------------------------------- the column kernel's timeline

TL_POINTS = {0: "producer: layer top", 1: "producer: barrier seen", 2: "producer: ids loaded",
             3: "consumers: activations formed", 4: "producer: down copies issued",
             5: "consumers: layer top", 6: "consumers: met the helper",
             7: "consumers: x operand built", 8: "consumers: first stage landed",
             9: "consumers: thread 0 done with gate/up", 10: "consumers: every warp done with gate/up",
             11: "consumers: planes built", 12: "consumers: down stages consumed",
             13: "consumers: partials written", 14: "consumers: arrived",
             15: "helper: owner's sums and shared scalar done",
             52: "helper: previous layer's arrivals complete",
             53: "producer: stage counts published", 54: "producer: first ring slot claimed"}


def timeline_summary(tl: np.ndarray) -> dict:
    """Medians over CTAs and the inner layers of the column kernel's per-layer stamps, in us after
    the consumers' layer top (clock64 within a CTA, converted with that CTA's own cycles per ns):
    the named points, when each of the layer's first ring stages was issued and found full, and
    the device-wide arrival count in globaltimer ns after the layer's last arrival."""
    t = tl.astype(np.int64)
    C, L, _ = t.shape
    lo, hi = (2, L - 2) if L > 6 else (1, L - 1)
    rate = (t[:, hi, 5] - t[:, lo, 5]) / np.maximum(t[:, hi, 56] - t[:, lo, 56], 1)  # cycles/ns
    base = t[:, lo:hi, 5]

    def rel(k):
        return (t[:, lo:hi, k] - base) / rate[:, None] / 1e3

    def stat(d):
        return {"median_us": round(float(np.median(d)), 3),
                "p10_us": round(float(np.percentile(d, 10)), 3),
                "p90_us": round(float(np.percentile(d, 90)), 3)}

    pts = {name: stat(rel(k)) for k, name in TL_POINTS.items()}
    stages = []
    for i in range(12):
        got = t[:, lo:hi, 16 + i]
        if not (got > 0).all():
            break
        waited = t[:, lo:hi, 40 + i] > 0
        wait_us = float(np.median(rel(40 + i)[waited])) if waited.any() else None
        stages.append({"stage": i, "issued_us": round(float(np.median(rel(28 + i))), 3),
                       "wait_from_us": None if wait_us is None else round(wait_us, 3),
                       "full_us": round(float(np.median(rel(16 + i))), 3)})
    layer_us = (t[:, lo + 1:hi + 1, 5] - t[:, lo:hi, 5]) / rate[:, None] / 1e3
    arrive = t[:, :, 57]
    last = arrive.max(axis=0)
    seen_after = (t[:, lo + 1:hi + 1, 59] - last[None, lo:hi]) / 1e3
    helper_after = (t[:, lo + 1:hi + 1, 58] - last[None, lo:hi]) / 1e3
    spread = (last[lo:hi] - np.median(arrive[:, lo:hi], axis=0)) / 1e3
    slow = np.bincount(np.argmax(arrive[:, lo:hi], axis=0), minlength=C)
    return {"ctas": C, "layers": L, "inner_layers": [lo, hi],
            "sm_ghz_median": round(float(np.median(rate)), 3),
            "layer_us": {"median": round(float(np.median(layer_us)), 3),
                         "p10": round(float(np.percentile(layer_us, 10)), 3),
                         "p90": round(float(np.percentile(layer_us, 90)), 3)},
            "points_after_consumer_layer_top": pts, "stages": stages,
            "barrier": {"producers_see_after_last_arrival_us": round(float(np.median(seen_after)), 3),
                        "helpers_see_after_last_arrival_us": round(float(np.median(helper_after)), 3),
                        "last_arrival_after_median_arrival_us": round(float(np.median(spread)), 3),
                        "ctas_most_often_last": [int(c) for c in np.argsort(-slow)[:8]],
                        "times_last": [int(slow[c]) for c in np.argsort(-slow)[:8]]}}


def run_timeline(args, shape: Shape):
    """The column kernel from the timeline build (libmoe_decode_timeline.so), stamped per CTA
    and layer; prints a summary of the last of --steps steps (not a throughput figure)."""
    import torch

    from quantized_moe_expert_dequant_gb300 import binding as Bn
    from quantized_moe_expert_dequant_gb300 import build as B

    B.build(timeline=True)
    Bn.use_timeline_build()
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    L, S = shape.layers, args.input_sets
    layers = [Bn.synth_layer_device(shape, l) for l in range(L)]
    mode = Bn.KERNELS_COLUMNS_AHEAD if args.kernels == "columns-ahead" else Bn.KERNELS_COLUMNS
    stack = Bn.MoeStack(layers, max_tokens=1, kernel_mode=mode)
    sets = []
    for i in range(S):
        x, ids, sc, r0 = input_set(shape, 1, i)
        conv = lambda a, dt: (torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(dt)
                              if dt == torch.bfloat16 else torch.from_numpy(np.ascontiguousarray(a)))
        sets.append((conv(x, torch.bfloat16).to(device), conv(ids, torch.int32).to(device),
                     conv(sc, torch.float32).to(device), conv(r0, torch.bfloat16).to(device),
                     torch.empty((1, shape.din), dtype=torch.float32, device=device)))
    stream = torch.cuda.current_stream(device)
    for i in range(args.warmup + args.steps):
        stack.step(*sets[i % S], stream=stream)
    torch.cuda.synchronize(device)
    assert stack.get_error() == 0
    tl = stack.timeline()
    if args.timeline_out:
        np.save(args.timeline_out, tl)
    line = {"timeline": shape.name, "kernel": "cols_kernel (timeline build)",
            "ids_known_ahead": mode == Bn.KERNELS_COLUMNS_AHEAD, **timeline_summary(tl)}
    print(json.dumps(line), flush=True)
    stack.close()
    return 0


# ---------------------------------------------------------------- the dense bf16 GEMV workload

GEMV_METRIC = "dense bf16 decode GEMV GB/s (weights streamed), 1 GB300"


def run_gemv(args):
    """A projection of "Measure attention projections instead of serving them, and record the
    amortisation trap" at --rows rows: one launch streams R distinct copies of the weight matrix,
    R chosen so that a launch moves at least 1 GiB (the page's rule: never time cache-resident
    weights), all rows multiplied by one seeded input."""
    import torch

    from quantized_moe_expert_dequant_gb300 import binding as Bn
    from quantized_moe_expert_dequant_gb300.workloads import GEMV

    rank, world, local = dist_setup("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    g, m = GEMV[args.gemv], args.rows
    if not 1 <= m <= 32:
        raise SystemExit("--rows must be in 1..32")
    R = -(-(1 << 30) // g.weight_bytes())
    W1 = synth.dense_weight(g.seed, g.n_out, g.n_in)
    x_host = synth.dense_input(g.seed, m, g.n_in)
    w1 = torch.from_numpy(W1.view(np.int16)).view(torch.bfloat16).to(device)
    W = w1.unsqueeze(0).repeat(R, 1, 1).contiguous()          # R distinct copies in HBM
    x = torch.from_numpy(x_host.view(np.int16)).view(torch.bfloat16).to(device)
    y = torch.empty((R, m, g.n_out), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    bus = None
    try:
        bus = torch.cuda.get_device_properties(device).pci_bus_id
    except AttributeError:
        bus = None
    sampler = ClockSampler(bus if bus else str(local))
    for _ in range(args.warmup):
        Bn.gemv_bf16(W, x, y, stream=stream)
    torch.cuda.synchronize(device)
    barrier(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        Bn.gemv_bf16(W, x, y, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize(device)
    barrier(device)
    ms = max_over_ranks(e0.elapsed_time(e1), device) / args.steps
    wbytes = R * g.weight_bytes()
    io = R * m * g.n_out * 4 + m * g.n_in * 2
    value = world * wbytes / (ms * 1e-3) / 1e9
    # end to end: pinned host input in, launch, host result out, every step
    xh = torch.from_numpy(x_host.view(np.int16)).view(torch.bfloat16).pin_memory()
    yh = torch.empty((R, m, g.n_out), dtype=torch.float32).pin_memory()
    e2e_steps = max(args.steps // 4, 5)
    torch.cuda.synchronize(device)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        x.copy_(xh, non_blocking=True)
        Bn.gemv_bf16(W, x, y, stream=stream)
        yh.copy_(y, non_blocking=True)
        torch.cuda.synchronize(device)
    e2e_s = max_over_ranks(time.perf_counter() - t0, device)
    clocks = sampler.stop()
    err = float((y[0].cpu().double() - y[R - 1].cpu().double()).abs().max())
    assert err == 0.0, "copies of one matrix gave different results"
    peaks = measured_peaks()
    peak = peaks["hbm_gbs"] if peaks else 6800.0
    note = "of measured" if peaks else "of fallback"
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import oracle as O
        n = 0
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < min(args.cpu_seconds, 10.0):
            O.gemv_bf16(W1, x_host)
            n += 1
        spent = time.perf_counter() - t0
        cpu = {"value": n * g.weight_bytes() / spent / 1e9, "unit": "GB/s", "cores": 1,
               "kind": "oracle",
               "sample": f"{n} products of one {g.n_out}x{g.n_in} matrix with {m} rows through "
                         f"the single-threaded fp64 oracle in {spent:.1f} s"}
    kernel = "gemv_cc_kernel" if m <= 4 else "gemv_mma_kernel"
    line = {
        "metric": GEMV_METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded bf16 weights and inputs)",
        "config": {"workload": g.name, "n_out": g.n_out, "n_in": g.n_in, "rows": m,
                   "matrices_per_launch": R, "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: {wbytes / 1e9:.2f} GB of distinct weight "
                         f"copies per launch"},
        "roofline": {"kernel": kernel, "bound": "hbm", "achieved": (wbytes + io) / (ms * 1e-3) / 1e9,
                     "peak": peak, "unit": "GB/s", "frac": (wbytes + io) / (ms * 1e-3) / 1e9 / peak,
                     "traffic": None, "bytes_per_launch": wbytes + io, "us_per_launch": ms * 1e3,
                     "note": note + " (copy peak)"},
        "cpu_baseline": cpu,
        "e2e": {"value": world * wbytes * e2e_steps / e2e_s / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": m * g.n_in * 2, "d2h_bytes_per_step": R * m * g.n_out * 4},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(ALL), default=DEFAULT_WORKLOAD)
    ap.add_argument("--tokens", type=int, default=1)
    ap.add_argument("--kernels", choices=["auto", "fused", "separate", "columns", "columns-ahead",
                                          "mma", "pool"],
                    default="auto",
                    help="fused: one persistent kernel per step (row split, two device-wide "
                         "barriers per layer); separate: kernel A and kernel B per layer; "
                         "columns: one persistent kernel per step with the column split (one "
                         "barrier per layer); mma: the tensor-core batch kernels (five launches "
                         "per layer); pool: the row split with each slot's output kept apart and "
                         "the page's tail association; auto: the column split for one token where it runs (no "
                         "folded norm, din <= 4096), the tensor-core kernels for batches of up to "
                         "64 tokens and 256 slots, else the row split.  columns-ahead: the column "
                         "split with every layer's ids treated as inputs known before the step "
                         "(the weight stream runs on into the next layer; not the decode "
                         "dependency)")
    ap.add_argument("--input-sets", type=int, default=4)
    ap.add_argument("--samples", type=int, default=10,
                    help="timed samples after the K steps (at least 10), each of at least 5 "
                         "replays and about 100 ms")
    ap.add_argument("--ab", choices=["fused", "separate", "columns", "columns-ahead", "mma", "pool"],
                    default=None,
                    help="also time this kernel mode, its samples alternating with the main "
                         "mode's (A/B on the same box and weights)")
    ap.add_argument("--chain-norm", action="store_true",
                    help="fold the next layer's RMSNorm in: layer l >= 1 reads RMSNorm(out of "
                         "layer l - 1) instead of its own x")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="run only the first N layers of the workload (profiling runs)")
    ap.add_argument("--gemv", choices=sorted(GEMV_NAMES), default=None,
                    help="measure the dense bf16 decode GEMV of this projection instead")
    ap.add_argument("--rows", type=int, default=1, help="rows (tokens) of the --gemv product")
    ap.add_argument("--timeline", action="store_true",
                    help="instead of timing, run the column kernel from the timeline build and "
                         "print where a layer's time goes (per-CTA, per-layer stamps)")
    ap.add_argument("--timeline-out", default=None, help="also save the raw stamps (.npy)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.gemv:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the GEMV workload has no "
                              "reference arm; its oracle baseline is in the line's cpu_baseline"}))
            return 0
        return run_gemv(args)
    shape = ALL[args.workload]
    single = shape.layers == 1
    if args.layers:
        shape = shape.with_(layers=args.layers, name=f"{shape.name} (first {args.layers} layers)")
    elif single:
        # one layer: a graph over R distinct weight replicas, R >= 48 and >= 1 GB of selected
        # weights per timed step, so that neither launch overhead nor L2 residency inflates the rate
        per = per_token_layer_weight_bytes(shape)
        R = max(48, -(-(1 << 30) // per))
        shape = shape.with_(layers=R, name=f"{shape.name}, {R} distinct replicas per step")
    args.single_layer = single and not args.layers
    if args.impl == "reference":
        return run_reference(args, shape)
    if args.timeline:
        return run_timeline(args, shape)
    return run_ours(args, shape)


if __name__ == "__main__":
    sys.exit(main())
