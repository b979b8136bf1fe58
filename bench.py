"""Benchmark: fused in-place QK RMSNorm + RoPE on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload all|NAME] [--impl ours|reference]

One step = one call of the fused op (qknr_apply, one kernel launch) over the
whole workload with inputs resident in HBM. Between timed steps the call
rotates over input replicas totalling at least 4x the L2 size, so no step
finds its inputs in L2. Rank 0 prints one JSON line.

By default every configuration runs (tiny, dit, mha_neox, gqa, fused_qkv),
one after another on the same GPU, each with its own W warm-up and K timed
steps. The line's headline is fused_qkv, the largest configuration;
``per_config`` carries every configuration's value, time per step and its
spread, roofline, clocks and CPU baseline. ``--workload NAME`` runs one.

Setup reads every input replica once with a torch reduction, so that no timed
launch pays the first kernel access to freshly copied memory. Timing: the
first warm-up step runs alone, then a synchronize and a barrier;
the other warm-up steps are enqueued back to back and the timed region's start
event is recorded right behind them, so the GPU is busy when it starts. K
steps follow, then an end event, a synchronize and a barrier; the time is the
maximum over ranks. The spread of the time per step comes from ten
further runs of K steps behind the timed region when K < 1000, else from
ten segments of it (an event between two launches costs the second its
programmatic overlap, so the timed region itself holds only two events).

Metric: effective HBM bandwidth = algorithmic bytes / time, where algorithmic
bytes = read + write of every Q/K head, one fp32 cos|sin row and one position
per token, and the two weight vectors; also heads/s and the fraction of the
measured HBM copy bandwidth.

The line also carries: the roofline object (DRAM read and write bytes of a
steady-state launch from the ncu summary in profiles/, while its source hash
matches the kernel's code, beside the algorithmic reads and writes), SM clocks
sampled around the timed region, the end-to-end leg through qknr_apply_host
from pinned host memory on the headline configuration (direct mode; staged
mode beside it), and the CPU baseline: the oracle on one core and on every
core.

--impl reference times the double-precision CPU oracle (the reference
implementation here: there is no runnable upstream code) on every host core,
each step a bounded sample of tokens of the same workload (the headline's by
default), and prints the same config dict as this arm.

Other options: --tokens N (decode-sized calls), --graph (replays of a CUDA
graph of calls), --inputs-ready (calls that set QKNR_INPUTS_READY), --variant
unfused (the two-kernel chain), --tune (qknr_tune picks each configuration's
launch first), --kernel register|ring (force one of the two kernels instead
of the library's rule), --ceiling (torch's own in-place elementwise kernel at
the same bytes).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import time
from typing import Dict, List, Optional

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "fused QK-RMSNorm+RoPE effective HBM GB/s (% of GB300 peak) and heads/sec"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
KERNEL_NAMES = {"register": "qknr_fused_kernel", "ring": "qknr_ring_kernel"}
# every configuration of the benchmark, small to large; the headline is the
# largest one that fits one GPU
CONFIGS = ["tiny", "dit", "mha_neox", "gqa", "fused_qkv"]
HEADLINE = "fused_qkv"


# ------------------------------------------------------------------ environment
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def init_dist(world: int, backend: str):
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
        return dist
    return None


def max_over_ranks(dist, value: float, device) -> float:
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


def measured_peaks() -> Dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


# device-code files each kernel is built from (a profile's counters stay valid
# while these are unchanged)
KERNEL_SOURCES = {
    "qknr_fused_kernel": ["qknr_math.cuh", "qknr_kernel.cuh"],
    "qknr_ring_kernel": ["qknr_math.cuh", "qknr_kernel.cuh", "qknr_ring_kernel.cuh"],
}


def code_tokens(text: str) -> str:
    """C/C++ source without comments and with whitespace collapsed: what the
    compiler sees (the kernel sources hold no comment markers inside string
    literals)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(kernel: str = "qknr_fused_kernel", read=None) -> str:
    """sha256 over the code (comments and layout ignored) of the files the
    kernel is built from; ``read(name)`` may supply another version's text."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "qk_rmsnorm_rope_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        if read is None:
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                text = f.read()
        else:
            text = read(name)
        h.update(name.encode() + b"\0" + code_tokens(text).encode())
    return h.hexdigest()


def profiled_traffic(kernel: str, workload: str) -> Optional[Dict[str, float]]:
    """DRAM bytes per launch from the committed ncu summary for this kernel and
    workload, if it was taken on the current kernel sources; else None.

    The summary gives the steady-state launch: the second of two back-to-back
    launches captured without cache flushes, so its writes include the lines
    the launch before it left dirty in L2 (what every launch of the timed loop
    pays) and miss those it leaves dirty itself."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.txt")
    try:
        with open(path) as f:
            lines = f.read().splitlines()
    except OSError:
        return None
    fields = {}
    for ln in lines:
        if ":" in ln:
            k, v = ln.split(":", 1)
            fields[k.strip()] = v.strip()
    if kernel not in KERNEL_SOURCES or fields.get("source_sha256") != kernel_source_hash(kernel):
        return None
    try:
        rd = float(fields["dram_read_bytes_per_launch"])
        wr = float(fields["dram_write_bytes_per_launch"])
    except (KeyError, ValueError):
        return None
    return {"read": rd, "write": wr, "total": rd + wr}


def smi_id(device) -> str:
    """nvidia-smi selector for a torch device (its UUID, so that a restricted
    CUDA_VISIBLE_DEVICES still names the right board)."""
    try:
        u = str(torch.cuda.get_device_properties(device).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(device.index or 0)


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: str, period_ms: int = 50):
        self.index = index
        self.period_ms = period_ms
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)  # let the first samples land before timing starts

    def stop(self) -> Dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in out.splitlines():
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() in ("active", "1"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ our arm
class PreparedCall:
    """One qknr_apply call's arguments, built once (pointers of one replica)."""

    def __init__(self, q, dev: Dict[str, torch.Tensor], w: workloads.Workload, stream: int,
                 entry: str = "qknr_apply", inputs_ready: bool = False):
        T, n_qo, D = dev["q"].shape
        n_kv = dev["k"].shape[1]
        hs = dev["q"].stride(1) if n_qo > 1 else dev["k"].stride(1)
        self.fn = getattr(q.lib, entry)
        self.args = (dev["q"].data_ptr(), dev["k"].data_ptr(), dev["q_w"].data_ptr(),
                     dev["k_w"].data_ptr(), dev["cos_sin_cache"].data_ptr(),
                     dev["positions"].data_ptr(), T, n_qo, n_kv, D, w.rope_dim, int(w.is_neox),
                     dev["q"].stride(0), dev["k"].stride(0), hs, w.eps,
                     q.dtype_code(dev["q"].dtype, dev["positions"].dtype)
                     | (q.QKNR_INPUTS_READY if inputs_ready else 0), stream)
        self.q = q

    def __call__(self):
        rc = self.fn(*self.args)
        if rc != 0:
            raise self.q.QknrError(rc, self.q.qknr_last_error())


def config_of(w: workloads.Workload) -> Dict:
    """The workload a line measures: the same dict in both arms."""
    return {"workload": w.name, "shape": workloads.describe(w), "storage_dtype": w.dtype,
            "bytes_per_step": workloads.algorithmic_bytes(w),
            "heads_per_step": workloads.num_heads_total(w)}


def peak_hbm() -> tuple:
    peak = measured_peaks().get("hbm_gbs")
    return (float(peak), "measured") if peak else (FALLBACK_HBM_GBS, "fallback")


# An event recorded between two launches costs the second one its
# programmatic overlap with the first (measured on dit: 21.1 -> 24.6 us per
# step with an event after every step). So the timed region holds only its
# two boundary events. The spread of the time per step comes, for K >= this
# many steps, from ten segments of the timed region (ten events: at most
# 0.16% of its time); below it, from ten further runs of K steps right
# behind the timed region, each between two events like the timed one.
SEGMENTS_FROM = 1000
SPREAD_RUNS = 10


def _spread(per_step: List[float], over: str) -> Dict:
    per = sorted(per_step)
    n = len(per)
    pick = lambda f: per[min(n - 1, int(round(f * (n - 1))))]
    return {"p10": round(pick(0.1), 6), "p50": round(pick(0.5), 6), "p90": round(pick(0.9), 6),
            "unit": "ms per step", "over": over}


def timed_region(calls, n_rep: int, steps: int, warmup: int, stream, device, dist, graph=None,
                 replays_per_step: int = 1) -> Dict:
    """W warm-up steps, then exactly K timed steps, on ``stream``.

    The first warm-up step runs alone (first-use host work), then a full
    synchronize and a barrier. The other warm-up steps go out back to back
    and the timed region starts directly behind them on the same stream (its
    start event is recorded right after the last warm-up call, with no
    synchronize in between), so the GPU is never idle at its start. A
    synchronize and a barrier close it. Clocks are sampled from before the
    warm-up to after the region."""
    sampler = ClockSampler(smi_id(device))
    if graph is None:
        calls[0]()
    torch.cuda.synchronize()
    sampler.start()
    barrier(dist)
    torch.cuda.synchronize()
    if graph is None:
        for i in range(1, warmup):
            calls[i % n_rep]()
    else:
        for _ in range(warmup):
            graph.replay()
    segments = graph is None and steps >= SEGMENTS_FROM
    n_seg = SPREAD_RUNS if segments else 0
    seg_len = steps // n_seg if n_seg else 0
    nxt = [warmup]

    def run(n: int, bounds=None):
        if graph is not None:
            for _ in range(n // replays_per_step):
                graph.replay()
            return
        for i in range(n):
            calls[nxt[0] % n_rep]()
            nxt[0] += 1
            if bounds is not None and (i + 1) % seg_len == 0 and len(bounds) < n_seg:
                ev = torch.cuda.Event(enable_timing=True)
                ev.record(stream)
                bounds.append(ev)

    ev0 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    bounds = [ev0]
    run(steps, bounds if segments else None)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev1.record(stream)
    # the spread's further runs (K < SEGMENTS_FROM): not part of the timed region
    runs = []
    if not segments:
        prev = ev1
        for _ in range(SPREAD_RUNS):
            run(steps)
            ev = torch.cuda.Event(enable_timing=True)
            ev.record(stream)
            runs.append((prev, ev))
            prev = ev
    torch.cuda.synchronize()
    barrier(dist)
    clocks = sampler.stop()
    ms = ev0.elapsed_time(ev1)
    if segments:
        bounds.append(ev1)
        lens = [seg_len] * (n_seg - 1) + [steps - seg_len * (n_seg - 1)]
        spread = _spread([bounds[j].elapsed_time(bounds[j + 1]) / lens[j] for j in range(n_seg)],
                         f"{n_seg} segments of the timed steps")
    else:
        spread = _spread([ms / steps] + [a.elapsed_time(b) / steps for a, b in runs],
                         f"the timed run and {SPREAD_RUNS} further runs of {steps} steps right behind "
                         "it, each between two events")
    return {"ms": max_over_ranks(dist, ms, device), "spread": spread, "clocks": clocks}


def measure_config(q, args, w: workloads.Workload, rank: int, world: int, device, stream, dist,
                   *, headline: bool) -> Optional[Dict]:
    """One workload on this GPU: build the input replicas, time K steps,
    and (rank 0) assemble its numbers."""
    sh = stream.cuda_stream
    cpu = workloads.make_inputs(w)
    qk_bytes = 2 * (w.n_qo + w.n_kv) * w.num_tokens * w.head_dim
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    n_rep = max(1, math.ceil(4 * l2 / qk_bytes)) if qk_bytes < 4 * l2 else 1
    l2_resident = n_rep > 64          # decode-sized inputs: 64 replicas, mostly in L2
    n_rep = min(n_rep, 64)
    reps = [workloads.to_device(cpu, w, device) for _ in range(n_rep)]
    # The copies above go through the copy engines. Read every replica once on
    # the SMs, so that no timed launch pays the first kernel access to freshly
    # copied memory (address translation) that a model's q and k, just written
    # by the kernel before, would not pay. At least 4x L2 of other replicas'
    # traffic passes between this read and a replica's first timed use.
    for r in reps:
        for key in ("buffer", "q", "k", "positions", "cos_sin_cache", "q_w", "k_w"):
            if key in r:
                r[key].view(-1).sum() if r[key].is_contiguous() else r[key].sum()
    torch.cuda.synchronize()
    entry = "qknr_apply_unfused" if args.variant == "unfused" else "qknr_apply"
    launches_per_step = 2 if args.variant == "unfused" else 1
    tuned = None
    if args.tune and args.variant == "fused":
        # qknr_tune for this call shape (timed on the library's own scratch
        # buffers, before and outside the warm-up and the timed region)
        r0 = reps[0]
        tuned = q.tune(r0["q"], r0["k"], r0["q_w"], r0["k_w"], r0["cos_sin_cache"], r0["positions"],
                       is_neox=w.is_neox, stream=stream, inputs_ready=args.inputs_ready)
        torch.cuda.synchronize()
    calls = [PreparedCall(q, r, w, sh, entry, args.inputs_ready) for r in reps]
    algo = workloads.algorithmic_bytes(w)
    heads = workloads.num_heads_total(w)

    graph = None
    steps = args.steps
    if args.graph:
        # one graph of n_rep calls (one per replica), replayed: GPU time per
        # call without the host's launch rate (decode-sized calls)
        for c in calls:
            c()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            cs = torch.cuda.current_stream().cuda_stream
            gcalls = [PreparedCall(q, r, w, cs, entry, args.inputs_ready) for r in reps]
            for c in gcalls:
                c()
        graph.replay()
        torch.cuda.synchronize()
        steps = max(1, steps // n_rep) * n_rep
    t = timed_region(calls, n_rep, steps, args.warmup, stream, device, dist, graph, n_rep)

    e2e = None
    if headline:
        # end to end through the C ABI from pinned host buffers, every step
        e2e = run_e2e(q, cpu, w, device, stream, args.e2e_steps, dist, entry)

    if rank != 0:
        return None
    secs = t["ms"] / 1e3
    value = world * algo * steps / secs / 1e9
    peak, peak_src = peak_hbm()
    per_launch_s = secs / steps
    achieved = algo / per_launch_s / 1e9
    wm = q.work_map(w.num_tokens, w.n_qo, w.n_kv, w.head_dim, w.rope_dim, w.is_neox,
                    q.dtype_code(w.torch_dtype, w.pos_torch_dtype))
    kernel = KERNEL_NAMES.get(wm["kernel"], str(wm["kernel"]))
    if args.variant == "unfused":
        kernel = "qknr_fused_kernel<..., kOpNorm> + qknr_fused_kernel<..., kOpRope>"
        wm = {"kernel": "register (norm step, rope step)"}
    full_size = w.num_tokens == workloads.get(w.name).num_tokens
    traffic = profiled_traffic(kernel, w.name) if (args.variant == "fused" and full_size) else None
    out = {
        "value": round(value, 1), "ms_per_step": t["ms"] / steps, "ms_per_step_spread": t["spread"],
        "config": config_of(w),
        "setup": {"l2": (f"rotating {n_rep} input replicas ({n_rep * qk_bytes / 1e6:.1f} MB, L2-resident: "
                         "a latency measurement)" if l2_resident else
                         f"rotating {n_rep} input replicas ({n_rep * qk_bytes / 1e6:.0f} MB >= 4x L2)"
                         if n_rep > 1 else "inputs larger than 4x L2"),
                  "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                  "launch": (f"CUDA graph of {n_rep} calls, replayed" if args.graph
                             else "one C-ABI call per step from Python")
                            + (", QKNR_INPUTS_READY" if args.inputs_ready else "")
                            + (", work map chosen by qknr_tune" if tuned else ""),
                  "work_map": wm},
        "heads_per_s": world * heads * steps / secs,
        "pct_of_peak": round(100.0 * achieved / peak, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "peak_source": peak_src, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic["total"] if traffic else None,
                     "traffic_read": traffic["read"] if traffic else None,
                     "traffic_write": traffic["write"] if traffic else None,
                     "algorithmic_bytes": algo,
                     "algorithmic_read": workloads.algorithmic_read_bytes(w),
                     "algorithmic_write": workloads.algorithmic_write_bytes(w),
                     "kernel": kernel},
        "clocks": t["clocks"],
        "gpu_launches": steps * launches_per_step,
    }
    if e2e is not None:
        out["e2e"] = e2e
    if world == 1 and not args.no_cpu_baseline:
        budget = args.cpu_seconds if headline else max(1.0, args.cpu_seconds / 4)
        out["cpu_baseline"] = cpu_baseline(w, cpu, budget_s=budget)
    del reps, calls, graph
    torch.cuda.empty_cache()
    return out


PER_CONFIG_KEYS = ["value", "ms_per_step", "ms_per_step_spread", "heads_per_s", "pct_of_peak",
                   "roofline", "clocks", "gpu_launches", "cpu_baseline", "config", "setup"]


def run_ours(args, names: List[str], rank: int, world: int, local: int) -> Optional[Dict]:
    import qk_rmsnorm_rope_gb300 as q

    backend = "nccl" if torch.cuda.is_available() else "gloo"
    dist = init_dist(world, backend)
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    q.init(local)
    if args.kernel != "auto":
        q.set_tuning(kernel=args.kernel)
    stream = torch.cuda.current_stream(device)
    head = HEADLINE if HEADLINE in names else names[-1]
    results = {}
    for name in names:
        w = workloads.get(name)
        if args.tokens > 0:
            w = workloads.scaled(w, args.tokens)
        results[name] = measure_config(q, args, w, rank, world, device, stream, dist,
                                       headline=(name == head))
    if rank != 0:
        return None
    h = results[head]
    line = {
        "metric": METRIC, "value": h["value"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": h["ms_per_step"],
        "ms_per_step_spread": h["ms_per_step_spread"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": h["config"],
        "setup": h["setup"],
        "heads_per_s": h["heads_per_s"], "pct_of_peak": h["pct_of_peak"],
        "roofline": h["roofline"], "clocks": h["clocks"], "e2e": h.get("e2e"),
        "gpu_launches": h["gpu_launches"],
    }
    if "cpu_baseline" in h:
        line["cpu_baseline"] = h["cpu_baseline"]
    if args.variant == "unfused":
        line["variant"] = ("unfused baseline: RMSNorm kernel then RoPE kernel, in place "
                           "(value counts the fused op's algorithmic bytes)")
    if len(names) > 1:
        line["headline"] = f"{head}: the largest configuration; per_config holds every configuration"
        line["per_config"] = {n: {k: results[n][k] for k in PER_CONFIG_KEYS if k in results[n]}
                              for n in names}
    return line


def run_e2e(q, cpu, w, device, stream, steps: int, dist, entry: str = "qknr_apply") -> Dict:
    if entry == "qknr_apply":
        return run_e2e_host(q, cpu, w, device, stream, steps, dist)
    dev = workloads.to_device(cpu, w, device)
    call = PreparedCall(q, dev, w, stream.cuda_stream, entry)
    if w.fused_total_heads:
        h_src = [cpu["buffer"].pin_memory()]
        d_dst = [dev["buffer"]]
    else:
        h_src = [cpu["q"].pin_memory(), cpu["k"].pin_memory()]
        d_dst = [dev["q"], dev["k"]]
    h_pos = cpu["positions"].pin_memory()
    h_out = [torch.empty_like(t, device="cpu").pin_memory() for t in d_dst]
    h2d = sum(t.numel() * t.element_size() for t in h_src) + h_pos.numel() * h_pos.element_size()
    d2h = sum(t.numel() * t.element_size() for t in h_out)

    def step():
        for d, h in zip(d_dst, h_src):
            d.copy_(h, non_blocking=True)
        dev["positions"].copy_(h_pos, non_blocking=True)
        call()
        for h, d in zip(h_out, d_dst):
            h.copy_(d, non_blocking=True)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    barrier(dist)
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    secs = time.perf_counter() - t0   # host wall clock: what the caller waits for
    world = dist.get_world_size() if dist is not None else 1
    secs = max_over_ranks(dist, secs, device)
    algo = workloads.algorithmic_bytes(w)
    return {"value": round(world * algo * steps / secs / 1e9, 2), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "path": "pinned host -> qknr_apply (C ABI) -> pinned host, one stream"}


def run_e2e_host(q, cpu, w, device, stream, steps: int, dist) -> Dict:
    """End to end through qknr_apply_host: every step, q, k and positions start
    in pinned host memory and the results end there. The headline runs the
    direct mode (the kernel reads and writes the pinned buffers in place over
    NVLink-C2C, both directions at once); the staged mode (chunked copies to
    device buffers, overlapped with the kernels) is timed beside it. Each step
    transforms the host q/k in place (the values stay bounded: every step
    re-normalises them)."""
    dev = workloads.to_device(cpu, w, device)
    if w.fused_total_heads:
        hb = cpu["buffer"].clone().pin_memory()
        h_q, h_k = hb[:, :w.n_qo, :], hb[:, w.n_qo:w.n_qo + w.n_kv, :]
    else:
        h_q, h_k = cpu["q"].clone().pin_memory(), cpu["k"].clone().pin_memory()
    h_pos = cpu["positions"].clone().pin_memory()
    d_q, d_k, d_pos = dev["q"], dev["k"], dev["positions"]
    T, n_qo, D = d_q.shape
    n_kv = d_k.shape[1]
    hs = d_q.stride(1) if n_qo > 1 else d_k.stride(1)
    fn = q.lib.qknr_apply_host
    heads_b = 2 * D * (n_qo + n_kv) * T
    h2d = heads_b + h_pos.numel() * h_pos.element_size()
    d2h = heads_b
    world = dist.get_world_size() if dist is not None else 1
    algo = workloads.algorithmic_bytes(w)
    values = {}
    for mode in (q.QKNR_HOST_DIRECT, q.QKNR_HOST_STAGED):
        args = (h_q.data_ptr(), h_k.data_ptr(), dev["q_w"].data_ptr(), dev["k_w"].data_ptr(),
                dev["cos_sin_cache"].data_ptr(), h_pos.data_ptr(), d_q.data_ptr(), d_k.data_ptr(),
                d_pos.data_ptr(), T, n_qo, n_kv, D, w.rope_dim, int(w.is_neox), d_q.stride(0),
                d_k.stride(0), hs, w.eps, q.dtype_code(d_q.dtype, d_pos.dtype), 0, mode,
                stream.cuda_stream)

        def step():
            rc = fn(*args)
            if rc != 0:
                raise q.QknrError(rc, q.qknr_last_error())

        for _ in range(3):
            step()
        torch.cuda.synchronize()
        barrier(dist)
        t0 = time.perf_counter()
        for _ in range(steps):
            step()
        torch.cuda.synchronize()
        secs = time.perf_counter() - t0   # host wall clock: what the caller waits for
        secs = max_over_ranks(dist, secs, device)
        values[mode] = round(world * algo * steps / secs / 1e9, 2)
    return {"value": values[q.QKNR_HOST_DIRECT], "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "path": ("pinned host q, k, positions -> qknr_apply_host (C ABI), direct mode: one kernel "
                     "reads and writes the pinned host buffers in place over NVLink-C2C"),
            "staged_value": values[q.QKNR_HOST_STAGED],
            "staged_path": ("qknr_apply_host staged mode: chunked host-to-device copies, kernels and "
                            "device-to-host copies overlapping on two copy streams and the caller's "
                            "stream")}


# ------------------------------------------------------------------ CPU oracle
def _sample_inputs(cpu, idx):
    return {"q": cpu["q"][idx], "k": cpu["k"][idx], "q_w": cpu["q_w"], "k_w": cpu["k_w"],
            "cos_sin_cache": cpu["cos_sin_cache"], "positions": cpu["positions"][idx]}


def _sample_bytes(w, n_tok):
    return workloads.algorithmic_bytes(workloads.scaled(w, n_tok, cache_len=w.cache_len))


def host_cpu() -> str:
    """The host CPU's model and core count (lscpu, else /proc/cpuinfo)."""
    model = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name:"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            for ln in open("/proc/cpuinfo"):
                if ln.lower().startswith(("model name", "cpu part")):
                    model = ln.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    return f"{model or 'unknown'}, {os.cpu_count()} cores"


def cpu_baseline(w, cpu, budget_s: float = 10.0) -> Dict:
    """The oracle as it stands (one thread, double precision) on a bounded
    sample: consecutive token blocks of the workload until ~budget_s seconds."""
    import oracle
    T = w.num_tokens
    block = min(T, 512)
    done_tok, t_used = 0, 0.0
    start = 0
    while t_used < budget_s and done_tok < 1024 * T:
        idx = torch.arange(start, start + block) % T
        sub = _sample_inputs(cpu, idx)
        t0 = time.perf_counter()
        oracle.apply(sub["q"], sub["k"], sub["q_w"], sub["k_w"], sub["cos_sin_cache"],
                     sub["positions"], is_neox=w.is_neox, eps=w.eps)
        t_used += time.perf_counter() - t0
        done_tok += block
        start = (start + block) % T
    value = _sample_bytes(w, done_tok) / t_used / 1e9
    return {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{done_tok} tokens of {w.name} in blocks of {block} ({t_used:.1f} s, "
                      f"double precision, single thread)",
            "heads_per_s": done_tok * (w.n_qo + w.n_kv) / t_used, "host": host_cpu(),
            "all_cores": cpu_baseline_all_cores(w, cpu, budget_s / 2)}


def cpu_baseline_all_cores(w, cpu, budget_s: float) -> Dict:
    """The same oracle on every host core at once: one thread per core, each on
    its own token blocks (the oracle is C code called through ctypes, which
    releases the GIL), for about budget_s seconds of wall time."""
    import concurrent.futures
    import oracle
    oracle.load()
    n = max(1, os.cpu_count() or 1)
    T = w.num_tokens
    block = min(T, 128)
    stop = time.perf_counter() + budget_s

    def worker(i):
        done, start = 0, (i * block) % T
        while time.perf_counter() < stop and done < 1024 * T:
            idx = torch.arange(start, start + block) % T
            sub = _sample_inputs(cpu, idx)
            oracle.apply(sub["q"], sub["k"], sub["q_w"], sub["k_w"], sub["cos_sin_cache"],
                         sub["positions"], is_neox=w.is_neox, eps=w.eps)
            done += block
            start = (start + n * block) % T
        return done

    torch_threads = torch.get_num_threads()
    torch.set_num_threads(1)   # the parallelism is the threads below, not torch's
    t0 = time.perf_counter()
    with concurrent.futures.ThreadPoolExecutor(max_workers=n) as ex:
        done_tok = sum(ex.map(worker, range(n)))
    secs = time.perf_counter() - t0
    torch.set_num_threads(torch_threads)
    return {"value": round(_sample_bytes(w, done_tok) / secs / 1e9, 4), "unit": UNIT, "cores": n,
            "kind": "oracle",
            "sample": f"{done_tok} tokens of {w.name}, {n} threads on blocks of {block} "
                      f"({secs:.1f} s wall, double precision)"}


def run_reference(args, w: workloads.Workload, rank: int, world: int) -> Optional[Dict]:
    """Reference arm: the CPU oracle, each step a bounded token sample."""
    if rank != 0:
        return None
    import oracle
    oracle.load()
    cpu = workloads.make_inputs(w)
    T = w.num_tokens
    # size the per-step sample so K+W steps take about a minute
    probe = min(T, 64)
    t0 = time.perf_counter()
    sub = _sample_inputs(cpu, torch.arange(probe))
    oracle.apply(sub["q"], sub["k"], sub["q_w"], sub["k_w"], sub["cos_sin_cache"],
                 sub["positions"], is_neox=w.is_neox, eps=w.eps)
    per_tok = max((time.perf_counter() - t0) / probe, 1e-7)
    # every host core works on its own slice of each step's sample (the oracle
    # is C code called through ctypes, which releases the GIL)
    import concurrent.futures
    cores = max(1, os.cpu_count() or 1)
    torch.set_num_threads(1)   # the parallelism is the threads below, not torch's
    target = 60.0 / max(1, args.steps + args.warmup)
    n_tok = int(max(cores, min(T, cores * target / per_tok)))
    pool = concurrent.futures.ThreadPoolExecutor(max_workers=cores)

    def part(s0, n):
        idx = torch.arange(s0, s0 + n) % T
        sb = _sample_inputs(cpu, idx)
        oracle.apply(sb["q"], sb["k"], sb["q_w"], sb["k_w"], sb["cos_sin_cache"],
                     sb["positions"], is_neox=w.is_neox, eps=w.eps)

    block = 128   # small pieces: each one's output arrays stay small (page faults serialise)

    def step(i):
        s0 = (i * n_tok) % T
        starts = list(range(0, n_tok, block))
        list(pool.map(lambda a: part(s0 + a, min(block, n_tok - a)), starts))

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    secs = time.perf_counter() - t0
    pool.shutdown()
    sample_bytes = _sample_bytes(w, n_tok)
    value = sample_bytes * args.steps / secs / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w),
        "sample_tokens_per_step": n_tok,
        "heads_per_s": n_tok * (w.n_qo + w.n_kv) * args.steps / secs,
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "host": host_cpu(),
                         "sample": (f"{n_tok} consecutive tokens of {w.name} per step"
                                    + (" (the whole workload)" if n_tok == T else "")
                                    + f", in blocks of {block} over {cores} threads")},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_ceiling(args, w: workloads.Workload) -> Dict:
    """Context line: torch's own in-place elementwise kernel (x.mul_(1)) and
    out-of-place copy on bf16 buffers moving exactly this workload's
    algorithmic bytes per step, rotated over >= 4x L2 like the op's inputs:
    what a plain streaming read-modify-write reaches on this GPU."""
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    algo = workloads.algorithmic_bytes(w)
    n = max(1, algo // 4)                       # bf16 elements: 2 B read + 2 B written each
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    reps = max(1, math.ceil(4 * l2 / (2 * n))) if 2 * n < 4 * l2 else 1
    reps = min(reps, 64)
    xs = [torch.zeros(n, dtype=torch.bfloat16, device=device) for _ in range(reps)]
    ys = [torch.zeros(n, dtype=torch.bfloat16, device=device) for _ in range(reps)]

    def timed(fn):
        for i in range(args.warmup):
            fn(i)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(args.steps):
            fn(i)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / args.steps

    t_inplace = timed(lambda i: xs[i % reps].mul_(1.0))
    t_copy = timed(lambda i: ys[i % reps].copy_(xs[i % reps]))
    return {"ceiling": "torch elementwise kernels at this workload's byte count",
            "workload": w.name, "bytes_per_step": 4 * n, "replicas": reps,
            "inplace_mul_gbs": round(4 * n / t_inplace / 1e9, 1),
            "copy_gbs": round(4 * n / t_copy / 1e9, 1),
            "steps": args.steps, "warmup": args.warmup}


def main(argv: Optional[List[str]] = None) -> int:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="all", choices=["all"] + sorted(workloads.WORKLOADS),
                    help="all (default): every configuration, headline on the largest; or one of them")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=0,
                    help="run the workload with this many tokens instead (e.g. 1 for decode latency)")
    ap.add_argument("--ceiling", action="store_true",
                    help="print torch's in-place elementwise and copy throughput at this "
                         "workload's byte count instead (context, not the op)")
    ap.add_argument("--inputs-ready", action="store_true",
                    help="pass QKNR_INPUTS_READY (weights and positions not written by the previous kernel)")
    ap.add_argument("--graph", action="store_true",
                    help="time replays of a CUDA graph of calls (GPU time per call, no host launch rate)")
    ap.add_argument("--variant", default="fused", choices=["fused", "unfused"],
                    help="unfused: time the two-kernel RMSNorm-then-RoPE chain instead")
    ap.add_argument("--kernel", default="auto", choices=["auto", "register", "ring"],
                    help="force one of the two kernels (default: the library's measured rule)")
    ap.add_argument("--tune", action="store_true",
                    help="call qknr_tune for each configuration's shape first (the launch it picks "
                         "on scratch buffers is then used)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.steps < 1:
        ap.error("--steps must be at least 1")
    rank, world, local = dist_env()
    if world != args.gpus and world > 1:
        print(f"warning: WORLD_SIZE={world} but --gpus {args.gpus}", file=sys.stderr)
    names = CONFIGS if args.workload == "all" else [args.workload]
    if args.ceiling or args.impl == "reference":
        w = workloads.get(HEADLINE if args.workload == "all" else args.workload)
        if args.tokens > 0:
            w = workloads.scaled(w, args.tokens)
        if args.ceiling:
            line = run_ceiling(args, w) if rank == 0 else None
        else:
            line = run_reference(args, w, rank, world)
    else:
        line = run_ours(args, names, rank, world, local)
    if line is not None:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
