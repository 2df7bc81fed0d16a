#!/usr/bin/env python
"""Throughput of the Echo emulated all-reduce on one GB300.

Metric: bf16-input GB/s per emulated all-reduce call (P ranks x n bf16
elements per call / time per call), with the fraction of the HBM roofline.

A step is one pass of the whole hot path over the workload's call sequence.
The default workload is the largest: P=8 ranks of 1 GiB bf16 each (512 Mi
elements per rank, i.i.d. N(0, 0.02^2)), one compensated call with 4-bit codes
and g=128 (the pages quote their throughput figure for 1 GB messages), inputs
resident in HBM before the timed region.  Every call runs libecho.so's default
schedule through its C ABI: one kernel whose blocks each take a whole owner
tile (the push of every sender, the owner's sum and the gather); the two- and
three-kernel schedules of the same call, the persistent single kernel and the
default schedule with a bf16 compensator state are timed beside it.
The same line also times, under "also", the 8-bit variant of that workload,
the other workloads of 64 MiB per rank, and the latency of the smallest one
(P=2, n=4096), plain and replayed as a CUDA graph.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With --gpus N > 1 (one process per GPU under torchrun) every rank runs an
independent replica of the workload on its own GPU (the emulated all-reduce
has no cross-GPU exchange); the value is the work of all ranks over the
slowest rank's time.  Each call's buffers are checked and marshalled once
(echo.prepare_allreduce), outside the timed loops.  `--impl reference` times
the CPU oracle (the plain single-threaded restatement the GPU path is
checked against) on the host cores, its group positions split over all of
them, on a sample of the same workload.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "bf16-input GB/s per emulated all-reduce call; % of GB300 HBM roofline"
QUANTIZERS = {0: "zero-aware asymmetric", 1: "naive zero-point (ablation)",
              2: "symmetric grid (ablation)"}
G = 128
FALLBACK_HBM_GBS = 6800.0
SPEC_HBM_GBS = 7900.0
L2_BYTES = 126 * 2 ** 20


# ------------------------------------------------------------- byte model ----

def code_bytes_per_elem(bits: int, g: int = G) -> float:
    """Codes plus the 4-byte meta word of each g-element group."""
    return bits / 8 + 4 / g


def kernel_bytes(P: int, n: int, bits: int, compensated: bool, fused: bool,
                 state_bytes: int = 4, g: int = G) -> dict:
    """Algorithmic bytes each kernel must move per call (one call = P ranks x n).

    push:   reads the non-owned bf16 input, reads+writes its state, writes
            codes + meta:                  (P-1) n (2 + 2e + c)
    reduce: reads P-1 code tiles + meta, the owner's bf16 input and state
            (read+write), writes gather codes + meta:
                                           (P-1) n c + n (2 + 2e + c)
            (+ 2 P n when it also writes the P outputs)
    gather: reads gather codes + meta, writes P bf16 outputs:  n c + 2 P n
    e is the state's bytes per element (4 fp32, 2 bf16); the state terms drop
    out when uncompensated."""
    c = code_bytes_per_elem(bits, g)
    st = 2 * state_bytes if compensated else 0
    d = {"push": (P - 1) * n * (2 + st + c),
         "reduce": (P - 1) * n * c + n * (2 + st + c) + (2 * P * n if fused else 0)}
    if not fused:
        d["gather"] = n * c + 2 * P * n
    if P == 1:
        d["push"] = 0
    return d


def call_model_bytes(P, n, bits, compensated, fused, state_bytes=4, g=G):
    return sum(kernel_bytes(P, n, bits, compensated, fused, state_bytes, g).values())


def tile_kernel_bytes(P, n, bits, compensated, state_bytes=4, g=G):
    """Bytes the tile-fused kernel must move per call: the fused call's model
    without the owner's read of the push codes ((P-1) n c), which it decodes
    from the values it has just encoded: P n (2 + 2e) + (P-1) n c + n c + 2 P n."""
    c = code_bytes_per_elem(bits, g)
    st = 2 * state_bytes if compensated else 0
    return P * n * (2 + st) + (P - 1) * n * c + n * c + 2 * P * n


# ---------------------------------------------------------------- helpers ----

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s (MEASURED_PEAKS.json absent)"


KERNEL_SOURCES = {"push_kernel": "k_push.cu", "reduce_kernel": "k_reduce.cu",
                  "gather_kernel": "k_gather.cu", "call_kernel": "k_call.cu",
                  "tile_kernel": "k_tile.cu"}


def kernel_source_hash(kernel: str = "") -> str:
    """Hash of the code that defines `kernel` (its own source, the shared
    device headers and echo_internal.h), comments and blank space removed, so
    that host-only, comment-only or other kernels' changes keep a committed ncu
    figure valid and any change to the kernel's own code drops it.  Without a
    kernel name: every kernel source."""
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_error_compensated_gb300", "csrc")
    own = KERNEL_SOURCES.get(kernel)
    for name in sorted(os.listdir(csrc)):
        shared = name.endswith(".cuh") or name == "echo_internal.h"
        if not (shared or (name == own if own else name.startswith("k_"))):
            continue
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            code = f.read()
        code = re.sub(r"/\*.*?\*/", " ", code, flags=re.S)
        code = re.sub(r"//[^\n]*", " ", code)
        code = " ".join(code.split())
        h.update(name.encode() + b"\0" + code.encode())
    return h.hexdigest()[:16]


def traffic_key(workload: str, bits: int, g: int, state: str, quantizer: int, schedule: str) -> str:
    """The configuration an ncu traffic figure belongs to: everything that picks
    a different kernel instantiation or grid (the decay does neither)."""
    return f"{workload} bits={bits} g={g} state={state} quantizer={quantizer} schedule={schedule}"


def profiled_traffic(kernel: str, key: str, elements: int):
    """DRAM bytes per launch of `kernel` from the committed ncu summary of the
    configuration `key` (traffic_key), as (bytes, note); (None, None) when there
    is none or the kernel sources changed since it was taken.  A capture taken
    on a smaller case of the same configuration (`captured_elements` input
    elements per call instead of `elements`) is scaled by the element ratio,
    since every byte these streaming kernels move is proportional to it."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None, None
    ent = rec.get(key, {}).get(kernel)
    if not ent or ent.get("source_hash") != kernel_source_hash(kernel):
        return None, None
    dram = ent.get("dram_bytes_per_launch")
    cap = ent.get("captured_elements")
    if dram is None or not cap or cap == elements:
        return dram, None
    return int(dram * elements / cap), (f"scaled by {elements / cap:g} from an ncu capture of "
                                         f"{cap} input elements per call ({ent.get('capture')})")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 20 ms; each sample
    is stamped with the host clock on arrival, and only the samples inside
    the window marked around the timed region are reported."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, interval_ms: int = 20):
        import threading
        self.proc = None
        self.samples = []             # (host time, line)
        self.window = None
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            sel = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(interval_ms), *sel],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()
        time.sleep(0.1)               # let the first samples arrive

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.monotonic(), line))

    def mark(self, t0: float, t1: float):
        """The timed region's host-clock window (after synchronizing at both ends)."""
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.reader.join(timeout=5)
        parsed = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, line in self.samples:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                parsed.append((t, float(f[1]), float(f[2]),
                               [n for n, v in zip(names, f[5:9]) if v.lower() == "active"]))
            except ValueError:
                continue
        if not parsed:
            return None
        inside = parsed
        where = "all samples"
        if self.window is not None:
            t0, t1 = self.window
            inside = [p for p in parsed if t0 <= p[0] <= t1]
            where = "inside the timed region"
            if not inside:          # a region shorter than the interval: the next sample
                after = [p for p in parsed if p[0] >= t0]
                inside = after[:1] or parsed[-1:]
                where = "first sample after the timed region began"
        reasons = sorted({r for p in inside for r in p[3]})
        return {"sm_mhz": statistics.median(p[1] for p in inside),
                "sm_max_mhz": max(p[2] for p in parsed), "samples": len(inside),
                "sampled": where, "reasons": reasons}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world <= 1:
        return 0, 0, 1
    import torch
    import torch.distributed as dist
    rank = int(os.environ["RANK"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if backend == "nccl":
        torch.cuda.set_device(local)
    dist.init_process_group(backend)
    return rank, local, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    """The largest `value` over all ranks (the slowest rank's time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank_per_step: float, steps: int, world: int, max_ms: float) -> float:
    """Work of all ranks over the slowest rank's time, in GB/s."""
    return bytes_per_rank_per_step * steps * world / (max_ms / 1e3) / 1e9


# ------------------------------------------------------------- our arm -------

STATE_FMT = {"f32": 0, "bf16": 1, "f16": 2}            # ECHO_STATE_* codes
STATE_NAME = {"f32": "fp32", "bf16": "bf16", "f16": "fp16"}


def state_dtype(args):
    import torch
    return {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[args.state]


def set_state(echo, plan, args):
    """Applies --state/--decay to a plan; returns the state's bytes per element."""
    echo.echo_set_state(plan, STATE_FMT[args.state], args.decay)
    return 4 if args.state == "f32" else 2


def workload_sequence(args, number=None):
    """The call sequence a run times: the workload's own (one step of it), or,
    with --uncompensated, the same calls with no compensator state (the
    "4-bit, no compensation" row of the paper's Table 6); --calls keeps only
    the first calls."""
    import dataclasses
    from bit_error_compensated_gb300.workloads import call_sequence
    seq = call_sequence(args.workload if number is None else number, steps=1)
    if getattr(args, "uncompensated", False):
        seq = [dataclasses.replace(c, state="none") for c in seq]
    if number is None and args.calls:
        seq = seq[:args.calls]
    return seq


# --tile-form: the tile kernel's form (echo_set_tile_fused modes), as the
# config names it, and as the ncu traffic records key it.
TILE_MODE = {"auto": 1, "loop": 2, "parallel": 3}
TILE_FORM_NOTE = {"auto": "", "loop": " (rank loop)", "parallel": " (rank-parallel)"}
TILE_KEY = {"auto": "", "loop": "", "parallel": "_rp"}


def tile_form(args) -> str:
    return getattr(args, "tile_form", "auto")


def state_key(args) -> str:
    """The state format a measurement ran with ("none" when uncompensated)."""
    return "none" if getattr(args, "uncompensated", False) else args.state


def shape_of(number, tokens=None):
    """(name, P, n) of a workload, with the token count overridden for
    profiling runs on a smaller case of the same shape family."""
    from bit_error_compensated_gb300.workloads import WORKLOADS
    w = WORKLOADS[number]
    if not tokens or tokens == w.tokens:
        return w.name, w.P, w.n
    return f"{w.name}@{tokens}x{w.hidden}", w.P, tokens * w.hidden


def build_inputs(number, seq, distinct, device, tokens=None):
    import torch
    from bit_error_compensated_gb300.workloads import rank_inputs
    _, P, n = shape_of(number, tokens)
    xs = torch.empty((distinct, P, n), dtype=torch.bfloat16, device=device)
    for k in range(distinct):
        rank_inputs(number, seq[k], device, tokens=tokens or None, out=xs[k])
    return xs


def workload_config(args, world, seq):
    """The workload a line measures: the same dict for the GPU arm and for the
    reference arm (the oracle on the host cores), so the two can be paired."""
    from bit_error_compensated_gb300.workloads import WORKLOADS
    name, P, n = shape_of(args.workload, args.tokens)
    comp = sum(1 for c in seq if c.state != "none")
    sb = 0 if not comp else 4 if args.state == "f32" else 2
    calls = len(seq)
    distinct = calls
    return {"workload": name, "description": WORKLOADS[args.workload].description,
            "P": P, "n_per_rank": n, "bits": args.bits, "g": args.g,
            "calls_per_step": calls * max(1, getattr(args, "repeat", 1)),
            "compensated": comp == calls,
            "fused_gather": bool(args.fused), "quantizer": QUANTIZERS[args.quantizer],
            "schedule": ("one kernel, a block per owner tile" + TILE_FORM_NOTE[tile_form(args)]
                         if args.tile else
                         "one persistent kernel" if args.persistent else
                         "two kernels" if args.fused else "three kernels")
                        + (", CUDA graph of the call sequence" if args.graph else ""),
            "state": ({"format": STATE_NAME[args.state], "decay": args.decay} if comp
                      else {"format": "none"}),
            "io": "bf16 in/out, fp32 arithmetic, "
                  f"{args.bits}-bit codes, "
                  + (f"{STATE_NAME[args.state]} state" if comp else "no compensator state"),
            "l2": f"inputs distinct per call ({distinct} x {P * n * 2 >> 20} MiB resident); "
                  f"per-call working set {(P * n * (2 + 2 + 2 * sb)) >> 20} MiB > L2 "
                  f"({L2_BYTES >> 20} MiB)",
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU, P ranks emulated"}


def run_ours(args, rank, local, world):
    import torch
    from bit_error_compensated_gb300 import echo

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    number, bits, fused = args.workload, args.bits, args.fused
    wname, P, n = shape_of(number, args.tokens)
    seq = workload_sequence(args)
    calls = len(seq)
    xs = build_inputs(number, seq, calls, dev, args.tokens)
    out = torch.empty((P, n), dtype=torch.bfloat16, device=dev)
    g = args.g
    plan = echo.echo_plan(P, n, g, bits)
    echo.echo_set_fused(plan, fused)
    echo.echo_set_quantizer(plan, args.quantizer)
    echo.echo_set_persistent(plan, args.persistent)
    echo.echo_set_tile_fused(plan, TILE_MODE[tile_form(args)] if args.tile else 0)
    sb = set_state(echo, plan, args)
    sdt = state_dtype(args)
    states = {"fwd": echo.COMP_DEFAULT,
              "bwd": torch.zeros((P, n), dtype=sdt, device=dev) if any(
                  c.state == "bwd" for c in seq) else None,
              "none": None}
    out_rows = list(out)
    call_args = [(list(xs[k]), states[c.state]) for k, c in enumerate(seq)]
    # each call's buffers are checked and marshalled once, outside the timed loop
    prepared = [echo.prepare_allreduce(plan, ins, out_rows, comp) for ins, comp in call_args]

    reps = max(1, getattr(args, "repeat", 1))

    def step():
        for _ in range(reps):
            for call in prepared:
                call(stream)

    launches_per_call = (1 if args.persistent or args.tile
                         else (2 if fused else 3) - (1 if P == 1 else 0))
    parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        parity = first_calls_parity(args, xs, seq, prepared, out, stream)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if echo.echo_get_status(plan, stream) != 0:
        raise RuntimeError("device status word set during warm-up")
    if args.graph:
        # The whole call sequence captured once as a CUDA graph and replayed
        # as one step: the calls are the same, their launches cost less.
        graph = torch.cuda.CUDAGraph()
        gstream = torch.cuda.Stream(dev)
        gstream.wait_stream(stream)
        with torch.cuda.graph(graph, stream=gstream):
            for _ in range(reps):
                for call in prepared:
                    call(gstream)
        torch.cuda.synchronize(dev)
        step = graph.replay
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize(dev)

    # Timed region: K steps, CUDA events on the launching stream.
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    host_t0 = time.monotonic()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    evs[0].record(stream)
    for i in range(args.steps):
        step()
        evs[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark(host_t0, time.monotonic())
    barrier(world)
    clk = clocks.stop()
    ms = evs[0].elapsed_time(evs[-1])
    step_ms = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps))
    max_ms = max_over_ranks(ms, world)
    if echo.echo_get_status(plan, stream) != 0:
        raise RuntimeError("device status word set during the timed steps")

    bytes_in_per_call = P * n * 2
    value = whole_job_gbs(bytes_in_per_call * calls * reps, args.steps, world, max_ms)
    per_call_s = max_ms / 1e3 / (args.steps * calls * reps)
    compensated_calls = sum(1 for c in seq if c.state != "none")
    model = (compensated_calls * call_model_bytes(P, n, bits, True, fused, sb, g) +
             (calls - compensated_calls) * call_model_bytes(P, n, bits, False, fused, g=g)) / calls
    hbm, hbm_src = load_peaks()

    # Per-kernel durations: the same K steps again, with events around each
    # kernel of every call (this makes each launch stream-serialised).
    raw_us = kernel_event_times(echo, plan, [(ins, out_rows, comp) for ins, comp in call_args],
                                stream, args.steps)
    avg_us, kb_avg, per_kernel_frac = kernel_fracs(raw_us, P, n, bits, fused, sb, g,
                                                   compensated_calls, calls, args.persistent, hbm,
                                                   args.tile)
    dominant = max(avg_us, key=lambda k: avg_us[k])
    kbytes = kb_avg[dominant]
    achieved = kbytes / (avg_us[dominant] / 1e6) / 1e9
    kname = {"push": "push_kernel", "reduce": "reduce_kernel", "gather": "gather_kernel",
             "call": "call_kernel", "tile": "tile_kernel"}[dominant]
    schedule = ("tile" + TILE_KEY[tile_form(args)] if args.tile else "persistent" if args.persistent
                else "fused" if fused else "unfused")
    traffic, traffic_note = profiled_traffic(
        kname, traffic_key(shape_of(number)[0], bits, g, state_key(args), args.quantizer, schedule),
        P * n)
    roofline = {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1), "peak": hbm,
                "unit": "GB/s", "frac": round(achieved / hbm, 4), "traffic": traffic,
                "algorithmic_bytes_per_launch": int(kbytes), "avg_launch_us": round(avg_us[dominant], 2),
                "peak_source": hbm_src}
    if traffic_note:
        roofline["traffic_note"] = traffic_note

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(max_ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; shapes and distributions of the workload, no dataset)",
        "config": workload_config(args, world, seq),
        "hbm_roofline_frac": round(model / per_call_s / 1e9 / hbm, 4),
        "hbm_roofline_frac_spec": round(model / per_call_s / 1e9 / SPEC_HBM_GBS, 4),
        "model_bytes_per_call": int(model),
        "us_per_call": round(per_call_s * 1e6, 2),
        "step_ms": {"median": round(step_ms[len(step_ms) // 2], 4), "min": round(step_ms[0], 4),
                    "max": round(step_ms[-1], 4)},
        "per_kernel_us": {k: round(v, 2) for k, v in avg_us.items()},
        "per_kernel_frac": per_kernel_frac,
        "roofline": roofline,
        "gpu_launches": launches_per_call * calls * reps * args.steps,
        "clocks": clk,
    }
    if parity is not None:
        result["parity"] = parity

    if not args.no_e2e:
        result["e2e"] = run_e2e(args, echo, plan, xs, seq, states, dev, world)
        torch.cuda.empty_cache()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle's sample is gathered from the inputs already on the device
        result["cpu_baseline"] = cpu_baseline_oracle(args, budget_s=args.cpu_budget, xs=xs, seq=seq)
    if args.also:
        result["also"] = {}
        for spec in [v for v in args.also.split(",") if v]:
            num, b = parse_also(spec, bits)
            label = shape_of(num)[0] + (f" ({b}-bit codes)" if b != bits else "")
            result["also"][label] = time_other(echo, num, b, fused, dev, args)
        if not args.persistent and not args.tokens:
            # the same workload with the other schedules, for comparison
            del xs, call_args, prepared, out_rows, out
            torch.cuda.empty_cache()
            others = [("two kernels", True, False), ("separate gather kernel", False, False),
                      ("one kernel, a block per owner tile", True, True)]
            for label, f, t in others:
                if (f, t) != (fused, args.tile):
                    result["also"][f"{wname} ({label})"] = time_other(echo, number, bits, f, dev,
                                                                      args, tile=t)
            # the persistent single kernel, and the 2-byte compensator state in
            # the default schedule
            variants = [("persistent single kernel", {"persistent": True}),
                        ("bf16 compensator state", {"state": "bf16"})]
            for label, over in variants:
                if all(getattr(args, k) != v for k, v in over.items()) and not args.uncompensated:
                    result["also"][f"{wname} ({label})"] = time_other(
                        echo, number, bits, fused, dev, argparse.Namespace(**{**vars(args), **over}))
    del plan
    return result


def kernel_event_times(echo, plan, calls, stream, steps):
    """Average device time of each kernel of a call, in microseconds: `steps`
    passes over `calls` (a list of (ins, outs, comp)), with events recorded
    around every kernel (which serialises the launches)."""
    import torch
    ev_sets = []
    torch.cuda.synchronize()
    for _ in range(steps):
        for ins, outs, comp in calls:
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            for e in evs:
                e.record(stream)
            echo.echo_set_timing(plan, evs)
            echo.echo_allreduce(plan, ins, outs, comp, stream)
            ev_sets.append(evs)
    echo.echo_set_timing(plan, None)
    torch.cuda.synchronize()
    tot = {"push": 0.0, "reduce": 0.0, "gather": 0.0}
    for evs in ev_sets:
        tot["push"] += evs[0].elapsed_time(evs[1])
        tot["reduce"] += evs[1].elapsed_time(evs[2])
        tot["gather"] += evs[2].elapsed_time(evs[3])
    return {k: v / len(ev_sets) * 1e3 for k, v in tot.items()}


def kernel_fracs(avg_us, P, n, bits, fused, sb, g, comp_calls, calls, persistent, hbm, tile=False):
    """Per-kernel achieved GB/s over the byte model, as fractions of `hbm`, and
    the kernels that ran."""
    kb_comp = kernel_bytes(P, n, bits, True, fused, sb, g)
    kb_unc = kernel_bytes(P, n, bits, False, fused, g=g)
    if tile:
        kb_comp = {"tile": tile_kernel_bytes(P, n, bits, True, sb, g)}
        kb_unc = {"tile": tile_kernel_bytes(P, n, bits, False, g=g)}
        avg_us = {"tile": avg_us["push"]}
        ran = ["tile"]
    elif persistent:
        kb_comp = {"call": sum(kb_comp.values())}
        kb_unc = {"call": sum(kb_unc.values())}
        avg_us = {"call": avg_us["push"]}
        ran = ["call"]
    else:
        ran = [k for k in ("push", "reduce", "gather") if k in kb_comp and (k != "push" or P > 1)]
    kb = {k: (comp_calls * kb_comp[k] + (calls - comp_calls) * kb_unc[k]) / calls for k in ran}
    avg = {k: avg_us[k] for k in ran}
    frac = {k: round(kb[k] / (avg[k] / 1e6) / 1e9 / hbm, 4) for k in ran}
    return avg, kb, frac


def parse_also(spec: str, default_bits: int):
    """'4' -> (4, default bits); '3b8' -> workload 3 with 8-bit codes."""
    if "b" in spec:
        num, b = spec.split("b")
        return int(num), int(b)
    return int(spec), default_bits


def run_e2e(args, echo, plan, xs, seq, states, dev, world):
    """The same call sequence from pinned host memory: every call copies its
    inputs host->device and one of its P output rows (all P rows hold the same
    bits: the result every rank receives) device->host, inside the timed
    region.  Copies run on their own streams, double-buffered, so the copy of
    call k+1 overlaps call k."""
    import torch
    P, n = xs.shape[1], xs.shape[2]
    distinct = min(8, xs.shape[0])
    host_in = []
    for k in range(distinct):
        h = torch.empty((P, n), dtype=torch.bfloat16, pin_memory=True)
        h.copy_(xs[k])
        host_in.append(h)
    host_out = torch.empty((2, n), dtype=torch.bfloat16).pin_memory()
    dev_in = [torch.empty((P, n), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    dev_out = [torch.empty((P, n), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    s_comp = torch.cuda.current_stream(dev)
    s_h2d = torch.cuda.Stream(dev)
    s_d2h = torch.cuda.Stream(dev)
    ev_loaded = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_read = [torch.cuda.Event() for _ in range(2)]
    calls = len(seq)
    comps = [states[c.state] for c in seq]
    prepared = [[echo.prepare_allreduce(plan, list(dev_in[b]), list(dev_out[b]), comps[k])
                 for k in range(calls)] for b in range(2)]
    issued = [0]                                          # calls issued so far, all steps

    def step():
        for k in range(calls):
            b = issued[0] & 1                             # alternates across steps too
            reused = issued[0] >= 2
            with torch.cuda.stream(s_h2d):
                if reused:
                    s_h2d.wait_event(ev_done[b])          # dev_in[b] no longer read
                dev_in[b].copy_(host_in[k % distinct], non_blocking=True)
                ev_loaded[b].record(s_h2d)
            s_comp.wait_event(ev_loaded[b])
            if reused:
                s_comp.wait_event(ev_read[b])             # dev_out[b] copied out
            prepared[b][k](s_comp)
            ev_done[b].record(s_comp)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(ev_done[b])
                host_out[b].copy_(dev_out[b][0], non_blocking=True)
                ev_read[b].record(s_d2h)
            issued[0] += 1

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    barrier(world)
    t = time.perf_counter()
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize(dev)
    barrier(world)
    wall_ms = (time.perf_counter() - t) * 1e3
    max_ms = max_over_ranks(wall_ms, world)
    v = whole_job_gbs(P * n * 2 * calls, args.steps, world, max_ms)
    return {"value": round(v, 2), "unit": "GB/s", "h2d_bytes_per_step": P * n * 2 * calls,
            "d2h_bytes_per_step": n * 2 * calls, "ms_per_step": round(max_ms / args.steps, 3),
            "timing": "host wall clock around K steps, synchronized at both ends",
            "d2h": "one of the P output rows per call: every rank receives the same bits, "
                   "so one row is the call's whole result",
            "host_inputs": f"{distinct} distinct pinned input sets cycled over the {calls} calls"}


def time_other(echo, number, bits, fused, dev, args, tile=None):
    """Time another workload's call sequence (8 distinct inputs cycled, at
    least 20 calls): GB/s and the pipeline's fraction of the HBM roofline.
    For the launch-bound P=2, n=4096 workload also the time per call with the
    sequence replayed as a CUDA graph.  No parity here: the GPU tests check
    these workloads against the oracle."""
    import torch
    from bit_error_compensated_gb300.workloads import WORKLOADS
    w = WORKLOADS[number]
    seq = workload_sequence(args, number)
    distinct = min(8, len(seq))
    xs = build_inputs(number, seq, distinct, dev)
    out = torch.empty((w.P, w.n), dtype=torch.bfloat16, device=dev)
    plan = echo.echo_plan(w.P, w.n, args.g, bits)
    echo.echo_set_fused(plan, fused)
    echo.echo_set_quantizer(plan, args.quantizer)
    tile = args.tile if tile is None else tile
    echo.echo_set_persistent(plan, args.persistent)
    echo.echo_set_tile_fused(plan, TILE_MODE[tile_form(args)] if tile else 0)
    sb = set_state(echo, plan, args)
    bwd = torch.zeros((w.P, w.n), dtype=state_dtype(args), device=dev) if any(
        c.state == "bwd" for c in seq) else None
    comps = [{"fwd": echo.COMP_DEFAULT, "bwd": bwd, "none": None}[c.state] for c in seq]
    rows = [list(xs[k]) for k in range(distinct)]
    out_rows = list(out)
    stream = torch.cuda.current_stream(dev)
    launch_bound = w.P * w.n * 2 < (1 << 20)
    reps = max(3, -(-(2000 if launch_bound else 20) // len(seq)))

    prepared = [echo.prepare_allreduce(plan, rows[k % distinct], out_rows, comps[k])
                for k in range(len(seq))]

    def step(s=stream):
        for call in prepared:
            call(s)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / 1e3 / (reps * len(seq))

    per_call_s = timed(step)
    if echo.echo_get_status(plan, stream) != 0:
        raise RuntimeError(f"device status word set while timing {w.name}")
    hbm, _ = load_peaks()
    comp_calls = sum(1 for c in seq if c.state != "none")
    raw_us = kernel_event_times(echo, plan, [(rows[k % distinct], out_rows, comps[k])
                                             for k in range(len(seq))], stream, reps)
    k_us, _, k_frac = kernel_fracs(raw_us, w.P, w.n, bits, fused, sb, args.g, comp_calls, len(seq),
                                   args.persistent, hbm, tile and fused and not args.persistent)
    model = (comp_calls * call_model_bytes(w.P, w.n, bits, True, fused, sb, args.g) +
             (len(seq) - comp_calls) * call_model_bytes(w.P, w.n, bits, False, fused, g=args.g)) / len(seq)
    res = {"gbs": round(w.P * w.n * 2 / per_call_s / 1e9, 2), "us_per_call": round(per_call_s * 1e6, 2),
           "hbm_roofline_frac": round(model / per_call_s / 1e9 / hbm, 4), "bits": bits,
           "calls": len(seq) * reps, "calls_per_step": len(seq),
           "states": sorted({c.state for c in seq}),
           "per_kernel_us": {k: round(v, 2) for k, v in k_us.items()},
           "per_kernel_frac": k_frac}
    if launch_bound:
        res["note"] = ("launch-bound (a few KiB per call): the time per call is the figure; "
                       "us_per_call issues each call from Python, us_per_call_cuda_graph replays "
                       "a graph of the sequence repeated to about 200 calls (the GPU's own time)")
        graph = torch.cuda.CUDAGraph()
        gstream = torch.cuda.Stream(dev)
        gstream.wait_stream(stream)
        seqs = max(1, 200 // len(seq))
        with torch.cuda.graph(graph, stream=gstream):
            for _ in range(seqs):
                step(gstream)
        torch.cuda.synchronize(dev)
        res["us_per_call_cuda_graph"] = round(timed(graph.replay) * 1e6 / seqs, 2)
        del graph
    del prepared, plan, xs, bwd
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------- the oracle ----

def host_cpu_info() -> dict:
    """Usable host cores and the CPU model (lscpu, else /proc/cpuinfo)."""
    try:
        nproc = len(os.sched_getaffinity(0))
    except Exception:
        nproc = os.cpu_count() or 1
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        names = [ln.split(":", 1)[1].strip() for ln in out.splitlines()
                 if ln.strip().lower().startswith("model name")]
        model = "; ".join(dict.fromkeys(names)) or None
    except Exception:
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for ln in f:
                    if ln.lower().startswith(("model name", "cpu part")):
                        model = ln.split(":", 1)[1].strip()
                        break
        except Exception:
            pass
    return {"nproc": nproc, "cpu_model": model or "unknown"}


class OracleSample:
    """The oracle on a fixed sample of one workload's group positions (1/8 of
    them; 1/64 for the 1 GiB-per-rank workload).

    Each step is one call of the workload's sequence restricted to those
    positions -- exactly the oracle's work on them, since positions are
    independent -- with up to 4 distinct inputs cycled and the state carried.
    The inputs are the GPU arm's own (gathered from `xs` on the device) when
    given, else drawn from the workload's generator on the GPU when there is
    one (the same bits the GPU arm draws), else on the CPU (same distribution,
    other bits)."""

    def __init__(self, number, bits, g=G, mode=0, state_fmt=0, decay=1.0, tokens=None,
                 xs=None, seq=None):
        import numpy as np
        import torch
        from bit_error_compensated_gb300.workloads import call_sequence, rank_inputs
        name, P, n = shape_of(number, tokens)
        self.name, self.bits, self.P = name, bits, P
        self.opts = dict(mode=mode, state_fmt=state_fmt, decay=decay)
        seq = seq if seq is not None else call_sequence(number, steps=1)
        Gs = n // P // g
        frac = 64 if P * n * 2 > (4 << 30) else 8
        rng = np.random.default_rng(number)
        pos = np.sort(rng.choice(P * Gs, size=max(1, P * Gs // frac), replace=False))
        self.owners = (pos // Gs).astype(np.int32)
        idx = (pos[:, None] * g + np.arange(g)[None, :]).ravel()
        # one held-error array per compensator state of the sequence; an
        # uncompensated call reads and writes none
        self.states = [c.state for c in seq]
        self.e = {st: np.zeros((pos.size, P, g), np.float32)
                  for st in sorted(set(self.states) - {"none"})}
        self.inputs = []
        distinct = min(len(seq), 4)
        if xs is not None:
            src = "the GPU arm's inputs"
        elif torch.cuda.is_available():
            src = "the workload's generator on the GPU"
        else:
            src = "the workload's generator on the CPU"
        dev = xs.device if xs is not None else torch.device("cuda" if torch.cuda.is_available() else "cpu")
        idx_t = torch.from_numpy(idx).to(dev)
        self.idx_t = idx_t          # the sampled elements' indices within a rank
        for k in range(distinct):
            if xs is not None:
                x = xs[k % xs.shape[0]]
            else:
                x = rank_inputs(number, seq[k], dev, tokens=tokens or None)
            sel = x.index_select(1, idx_t).view(torch.int16).cpu().numpy().view(np.uint16)
            self.inputs.append(np.ascontiguousarray(sel.reshape(P, pos.size, g).transpose(1, 0, 2)))
            del x
        self.bytes_per_step = pos.size * P * g * 2
        self.sample = (f"each step: one call of {name} on a fixed 1/{frac} sample of its group "
                       f"positions ({pos.size} of {P * Gs}), {distinct} distinct input(s) cycled "
                       f"(from {src}), state carried")
        self.i = 0
        self.ties = 0          # exact rounding ties the oracle met (codes and zero points)

    def _chunk(self, x, e, a, b):
        import oracle
        r = oracle.group_positions(self.P, self.owners[a:b], self.bits, x[a:b],
                                   None if e is None else e[a:b], **self.opts)
        return r["ties"], r["y"]

    def step(self, pool=None, threads=1, want_y=False):
        """One call over all sampled positions: on this thread, or split into
        `threads` contiguous chunks run by `pool` (the oracle call releases
        the interpreter lock, so the chunks run on separate cores).  With
        want_y, returns the call's output at the sampled positions, [npos, g]
        bf16 bits."""
        import numpy as np
        x = self.inputs[self.i % len(self.inputs)]
        e = self.e.get(self.states[self.i % len(self.states)])
        npos = self.owners.size
        if pool is None or threads <= 1:
            parts = [self._chunk(x, e, 0, npos)]
        else:
            cuts = [npos * t // threads for t in range(threads + 1)]
            futs = [pool.submit(self._chunk, x, e, cuts[t], cuts[t + 1]) for t in range(threads)
                    if cuts[t + 1] > cuts[t]]
            parts = [f.result() for f in futs]
        self.ties += sum(t for t, _ in parts)
        self.i += 1
        return np.concatenate([y for _, y in parts]) if want_y else None


def oracle_sample(args, xs=None, seq=None):
    """OracleSample of the workload and options the GPU arm runs."""
    return OracleSample(args.workload, args.bits, args.g, args.quantizer, STATE_FMT[args.state],
                        args.decay, args.tokens, xs=xs, seq=seq)


def _time_steps(s, budget_s, pool=None, threads=1):
    s.step(pool, threads)                  # untimed first step
    steps, t = 0, time.perf_counter()
    while time.perf_counter() - t < budget_s or steps == 0:
        s.step(pool, threads)
        steps += 1
    return steps, time.perf_counter() - t


def first_calls_parity(args, xs, seq, prepared, out, stream, calls=2):
    """The first `calls` calls of the timed configuration, from its fresh state,
    against the oracle on the sampled group positions of OracleSample: every
    rank's output there, bit for bit.  A later call's output depends on the
    state the earlier calls left, so the state is checked through it."""
    from concurrent.futures import ThreadPoolExecutor
    import numpy as np
    import torch
    s = oracle_sample(args, xs, seq)
    threads = host_cpu_info()["nproc"]
    P, npos, g = s.P, s.owners.size, args.g
    mismatches = compared = 0
    with ThreadPoolExecutor(threads) as pool:
        for k in range(calls):
            prepared[k % len(prepared)](stream)
            if out.is_cuda:
                torch.cuda.synchronize(out.device)
            got = out.index_select(1, s.idx_t).view(torch.int16).cpu().numpy().view(np.uint16)
            want = s.step(pool, threads, want_y=True).reshape(1, npos * g)
            mismatches += int(np.count_nonzero(got != want))
            compared += got.size
    return {"calls": calls, "sampled_groups": npos, "outputs_compared": compared,
            "output_mismatches": mismatches, "exact_rounding_ties": s.ties,
            "what": "the first calls of the timed configuration from its fresh state, every "
                    "rank's output at the sampled group positions against the oracle, bit for "
                    "bit (the later call's outputs depend on the state the first one left)"}


def cpu_baseline_oracle(args, budget_s=12.0, xs=None, seq=None):
    """The oracle as it stands (single-threaded code) on a sample of the
    workload, timed for about budget_s / 2 seconds on one host core and as long
    again with the sampled positions split over every usable core."""
    from concurrent.futures import ThreadPoolExecutor
    info = host_cpu_info()
    s = oracle_sample(args, xs, seq)
    steps1, sec1 = _time_steps(s, budget_s / 2)
    v1 = s.bytes_per_step * steps1 / sec1 / 1e9
    threads = info["nproc"]
    with ThreadPoolExecutor(threads) as pool:
        stepsN, secN = _time_steps(s, budget_s / 2, pool, threads)
    vN = s.bytes_per_step * stepsN / secN / 1e9
    return {"value": round(vN, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{stepsN} steps on {threads} threads, {steps1} on one; " + s.sample,
            "nproc": info["nproc"], "cpu_model": info["cpu_model"],
            "single_core": {"value": round(v1, 4), "cores": 1, "steps": steps1,
                            "seconds": round(sec1, 2)},
            "all_cores": {"value": round(vN, 4), "cores": threads, "steps": stepsN,
                          "seconds": round(secN, 2)},
            "exact_rounding_ties": s.ties, "ties_counted_over_calls": s.i}


def run_reference(args, rank, world):
    """`--impl reference`: the oracle on the host cores (its sampled group
    positions split over all of them), K timed steps of OracleSample after W
    warm-up steps, on the workload and options of the GPU arm."""
    from concurrent.futures import ThreadPoolExecutor
    seq = workload_sequence(args)
    info = host_cpu_info()
    threads = info["nproc"]
    s = oracle_sample(args, seq=seq)
    with ThreadPoolExecutor(threads) as pool:
        for _ in range(args.warmup):
            s.step(pool, threads)
        t = time.perf_counter()
        for _ in range(args.steps):
            s.step(pool, threads)
        sec = time.perf_counter() - t
    v = s.bytes_per_step * args.steps / sec / 1e9
    return {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(sec / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded; shapes and distributions of the workload, no dataset)",
            "config": workload_config(args, world, seq),
            "sample": s.sample,
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": s.sample, "nproc": info["nproc"],
                             "cpu_model": info["cpu_model"], "exact_rounding_ties": s.ties,
                             "ties_counted_over_calls": s.i},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# --------------------------------------------------- accuracy (Table 8) ----

def run_accuracy(args):
    """A synthetic stand-in for the paper's Table 6 / Table 8 comparisons, which
    need models and datasets: for each quantizer, with and without the
    compensator, run the workload's call sequence and measure, against the
    exact sum of the bf16 inputs (fp64),
      per_call_rel_rms  RMS error of one call's output / RMS of the exact sum
                        (mean over calls), and
      drift_rel_rms     RMS of the error accumulated over the whole sequence /
                        RMS of one call's exact sum,
    the quantity whose growth the compensator is meant to stop."""
    import torch
    from bit_error_compensated_gb300 import echo
    from bit_error_compensated_gb300.workloads import WORKLOADS, call_sequence, rank_inputs
    number, bits = args.workload, args.bits
    w = WORKLOADS[number]
    P, n = w.P, w.n
    seq = call_sequence(number, steps=1)
    if args.calls:
        seq = seq[:args.calls]
    dev = torch.device("cuda", 0)
    x = torch.empty((P, n), dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(x)
    rows = {}
    # (quantizer, compensated, state format, decay)
    variants = [(qz, comp, "f32", 1.0) for qz in (0, 1, 2) for comp in (True, False)]
    variants += [(0, True, "bf16", 1.0), (0, True, "f16", 1.0), (0, True, "f32", 0.9),
                 (0, True, "bf16", 0.9)]
    for qz, compensated, fmt, decay in variants:
        plan = echo.echo_plan(P, n, args.g, bits)
        echo.echo_set_quantizer(plan, qz)
        echo.echo_set_state(plan, STATE_FMT[fmt], decay)
        sdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[fmt]
        states = {}
        drift = torch.zeros(n, dtype=torch.float64, device=dev)
        rel, scale = [], None
        for c in seq:
            rank_inputs(number, c, dev, out=x)
            comp = None
            if compensated and c.state != "none":
                comp = states.setdefault(c.state, torch.zeros((P, n), dtype=sdt, device=dev))
            echo.echo_allreduce(plan, list(x), list(out), comp)
            exact = x.double().sum(0)
            err = out[0].double() - exact
            drift += err
            ex_rms = float(exact.square().mean().sqrt())
            scale = scale or ex_rms
            rel.append(float(err.square().mean().sqrt()) / ex_rms)
        if echo.echo_get_status(plan) != 0:
            raise RuntimeError("status word set")
        label = f"{QUANTIZERS[qz]}, {'compensated' if compensated else 'uncompensated'}"
        if fmt != "f32" or decay != 1.0:
            label += f" ({STATE_NAME[fmt]} state, decay {decay})"
        rows[label] = {
            "per_call_rel_rms": round(sum(rel) / len(rel), 6),
            "drift_rel_rms": round(float(drift.square().mean().sqrt()) / scale, 6)}
        del plan
    return {"workload": w.name, "bits": bits, "calls": len(seq), "results": rows}


# ------------------------------------------------------------------- main ----

def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=3,
                    help="1..5 (default 3: P=8, 1 GiB bf16 per rank, one call)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="profiling runs: the workload's shape with this many tokens per rank")
    ap.add_argument("--bits", type=int, default=4, choices=[4, 8])
    ap.add_argument("--g", type=int, default=G, choices=[64, 128, 256], help="elements per group")
    ap.add_argument("--unfused", action="store_true",
                    help="separate gather kernel (three kernels per call); by default the reduce "
                         "kernel writes the outputs itself")
    ap.add_argument("--fused", action="store_true", help=argparse.SUPPRESS)   # the default
    ap.add_argument("--persistent", action="store_true",
                    help="one persistent kernel per call instead of two or three")
    ap.add_argument("--two-kernels", action="store_true",
                    help="push then reduce, two kernels per call, instead of one kernel whose "
                         "blocks each take a whole owner tile (the default)")
    ap.add_argument("--tile-form", choices=["auto", "loop", "parallel"], default="auto",
                    help="the one-kernel schedule's form: chosen by size (default), the rank "
                         "loop, or rank-parallel blocks")
    ap.add_argument("--graph", action="store_true",
                    help="time replays of the call sequence captured as a CUDA graph")
    ap.add_argument("--quantizer", type=int, default=0, choices=[0, 1, 2],
                    help="0 zero-aware (the method), 1 naive zero-point, 2 symmetric grid")
    ap.add_argument("--state", choices=["f32", "bf16", "f16"], default="f32",
                    help="compensator state storage (bf16 or fp16 halve its traffic)")
    ap.add_argument("--uncompensated", action="store_true",
                    help="every call without compensator state (no state read or written)")
    ap.add_argument("--decay", type=float, default=1.0,
                    help="kept error = decay x revealed error (1 = plain error feedback)")
    ap.add_argument("--also", default="3b8,2,4,5,1",
                    help="other workloads to time, comma-separated, NbB for workload N with B-bit "
                         "codes ('' for none)")
    ap.add_argument("--repeat", type=int, default=1,
                    help="latency runs: each timed step issues the call sequence this many times "
                         "(with --graph, one graph holds them all), so that host-side launch "
                         "costs are spread over many calls")
    ap.add_argument("--calls", type=int, default=0,
                    help="time only the first N calls of the sequence (profiling runs)")
    ap.add_argument("--accuracy", action="store_true",
                    help="report output error and accumulated drift per quantizer instead of timing")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    args = ap.parse_args(argv)
    args.fused = not args.unfused
    args.tile = not (args.two_kernels or args.unfused or args.persistent)
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be at least 3")

    if args.accuracy:
        print(json.dumps(run_accuracy(args)), flush=True)
        return 0
    rank, local, world = dist_setup()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)), flush=True)
        return 0
    res = run_ours(args, rank, local, world)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
