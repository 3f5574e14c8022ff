#!/usr/bin/env python
"""SAMU mixer forward+backward benchmark on GB300 (one JSON line on rank 0).

One step = samu_forward + samu_backward (BF16 gradients) through the C ABI on
the B=1, L=32768, D=2048 workload (the metric's configuration), inputs
resident in HBM.  The step's launches are captured once as a CUDA graph and
replayed; L2 is flushed (256 MiB memset) before every timed step and each step
is timed with its own CUDA events; the memset is outside the timed events.
Per-kernel durations come from a second, eager pass with the library's own
events around every launch.  Alongside the device-timed value the line
carries:
  e2e          the same metric through the public Python API with host (pinned)
               inputs copied in and results copied out inside the timed region;
  roofline     the dominant kernel's algorithmic bytes / its average CUDA-event
               duration (events recorded by the library on the launching stream)
               against the measured HBM copy bandwidth;
  cpu_baseline the FP64 oracle timed on the host (rank 0, N=1) on a bounded sample;
  clocks       nvidia-smi samples taken during the timed region.

--impl reference times the oracle itself (CPU) on the same metric.
Multi-GPU (torchrun): every rank runs its own independent batch (weak scaling,
no collective on the data path); the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "SAMU mixer F+B ms & Mtok/s (B1,L32K,D2048); achieved HBM GB/s vs GB300 peak"
UNIT = "Mtok/s"
DEFAULT_WORKLOAD = "width_2048"
FALLBACK_HBM_GBS = 6800.0
FLUSH_BYTES = 256 << 20
WARM_S = 0.3   # seconds of untimed graph replays before the timed region

# Bytes each launch must move, in units of B*L*D (one BF16 [B,L,D] tensor = 2 units):
#   controller forward: read x_sel (2)        forward maps: read w (2)
#   forward replay: read w, write y (4)       backward maps: read dy (2)
#   backward main: read dy, w, write dw (6)   controller backward: read x_sel, write dx_sel (4)
# The step's algorithmic total (x_sel, w, dy read once; y, dx_sel, dw written) is
# 16 units; the maps launches' second reads of w and dy are the price of the
# two-launch scan and count towards the kernels, not towards the step.
KERNEL_BYTES_PER_BLD = {
    "samu_ctrl_fwd_kernel": 2.0, "samu_fwd_maps_kernel": 2.0, "samu_fwd_replay_kernel": 4.0,
    "samu_bwd_maps_kernel": 2.0, "samu_bwd_main_kernel": 6.0, "samu_ctrl_bwd_kernel": 4.0,
}
STEP_BYTES_PER_BLD = 16.0
LAUNCHES_PER_RECORD = {"rglru_alpha_kernels": 2}


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=None)
    p.add_argument("--sweep", action="store_true",
                   help="time every workload family (one JSON line each) instead of the headline line")
    p.add_argument("--only", default=None, help="with --sweep: comma-separated workload names")
    p.add_argument("--compare-pages", action="store_true",
                   help="SAMU vs RG-LRU (with its gate projections) on the pages' comparison shapes with the "
                        "pages' timing protocol, one JSON line per shape")
    p.add_argument("--transition", choices=["closed_form", "chained"], default="closed_form",
                   help="form of the SAMU maps kernels' 16-token item transitions")
    return p.parse_args(argv)


def set_transition(args):
    from linear_recurrence_sequence_gb300 import api
    api.samu_set_chunk_transition(api.LRS_TRANSITION_CLOSED_FORM if args.transition == "closed_form"
                                  else api.LRS_TRANSITION_CHAINED)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def shard_seed(base_seed: int, rank: int) -> int:
    """Each rank draws its own independent batch (weak scaling)."""
    return base_seed + 1000 * rank


def reduce_max(value: float, world: int, device=None) -> float:
    """Max over ranks (timing); identity on a single process."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _code_only(text: str) -> str:
    """Source text with comments and whitespace runs removed: the hash below
    then changes with the code, not with its comments."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


# The sources the SAMU step's kernels and their launches are built from: the
# committed DRAM figures stay valid while these are unchanged.
STEP_SOURCES = ("linear_recurrence_sequence_gb300/csrc/samu_scan.cu",
                "linear_recurrence_sequence_gb300/csrc/samu_ctrl.cu",
                "linear_recurrence_sequence_gb300/csrc/abi.cu",
                "linear_recurrence_sequence_gb300/csrc/common.cuh",
                "linear_recurrence_sequence_gb300/csrc/kernels.cuh",
                "linear_recurrence_sequence_gb300/csrc/layout.cuh",
                "linear_recurrence_sequence_gb300/csrc/tmap.cuh",
                "include/samu.h")


def source_hash() -> str:
    h = hashlib.sha256()
    for rel in STEP_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(os.path.basename(rel).encode())
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def load_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def load_traffic(kernel: str, bld: int):
    """DRAM bytes per launch from a committed ncu capture, if the kernel sources
    are unchanged since it was taken; scaled by the units processed."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kernel]
    except Exception:
        return None
    if rec.get("source_sha") != source_hash():
        return None
    return float(rec["dram_bytes_per_bld"]) * bld


# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index_or_uuid):
        self.sel = device_index_or_uuid
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-i", str(self.sel)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self._t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_selector(device):
    import torch
    try:
        u = torch.cuda.get_device_properties(device).uuid
        return "GPU-" + str(u)
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        first = vis.split(",")[0] if vis else "0"
        return first if first.isdigit() else 0


# ---------------------------------------------------------------------------
def _oracle_inputs(B, L, D, seed):
    """Seeded SAMU sample widened for the oracle: (args, dy, dhT)."""
    from linear_recurrence_sequence_gb300 import synth
    inp = synth.samu_inputs(B, L, D, seed, h0=False)
    f64 = synth.bf16_bits_to_f64
    x, w, dy = f64(inp["x_sel"]), f64(inp["w"]), f64(inp["dy"])
    args = (x, w, inp["h0"], inp["reset"], inp["nu"], inp["theta"], inp["w_phi"], inp["w_r"],
            float(inp["a_phi"]), float(inp["a_r"]))
    return args, dy, inp["dhT"]


def _oracle_fb(args, dy, dhT):
    import oracle
    oracle.samu_forward(*args)
    oracle.samu_backward(*args, dy, dhT)


def oracle_sample_time(B, L, D, seed=0):
    """Seconds for one FP64 oracle forward+backward on a [B, L, D] SAMU sample."""
    args, dy, dhT = _oracle_inputs(B, L, D, seed)
    t0 = time.perf_counter()
    _oracle_fb(args, dy, dhT)
    return time.perf_counter() - t0


def host_cpu():
    """Host core count available to this process and the CPU model."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().startswith("Model name:"):
                model = ln.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if model is None:
        try:
            for ln in open("/proc/cpuinfo"):
                if ln.lower().startswith("model name"):
                    model = ln.split(":", 1)[1].strip()
                    break
        except Exception:
            pass
    return len(os.sched_getaffinity(0)), model or "unknown"


def cpu_baseline(D, target_s=12.0):
    """The oracle as it stands, on bounded samples of the workload (B=1, the
    workload's D): once on one thread, once on every host core with one
    independent sample per thread (the oracle is plain C called through
    ctypes, which releases the interpreter lock; the same kind of parallelism
    as the method's independent batch rows).  The all-cores rate is the
    reported value."""
    from concurrent.futures import ThreadPoolExecutor
    cores, model = host_cpu()
    t_small = oracle_sample_time(1, 256, D)
    per_tok = t_small / 256
    L1 = int(min(32768, max(512, 0.4 * target_s / max(per_tok, 1e-9))))
    L1 = max(512, (L1 // 256) * 256)
    t1 = oracle_sample_time(1, L1, D, seed=1)
    single = L1 / t1 / 1e6
    # every core: per thread `reps` forward+backward passes over its own
    # sample of Lp tokens, inputs drawn before the timed region
    Lp = max(256, min(4096, (int(0.5 / max(per_tok, 1e-9)) // 256) * 256))
    reps = max(1, int(0.6 * target_s / max(per_tok * Lp, 1e-9)))
    samples = [_oracle_inputs(1, Lp, D, 100 + k) for k in range(cores)]

    def work(k):
        for _ in range(reps):
            _oracle_fb(*samples[k])

    with ThreadPoolExecutor(max_workers=cores) as ex:
        t0 = time.perf_counter()
        list(ex.map(work, range(cores)))
        tp = time.perf_counter() - t0
    par = cores * reps * Lp / tp / 1e6
    del samples
    return {"value": par, "unit": UNIT, "cores": cores, "kind": "oracle", "cpu_model": model,
            "sample": f"{cores} threads, each {reps} FP64 forward+backward passes over its own B=1, L={Lp}, "
                      f"D={D} sample, {tp:.1f} s wall",
            "single_thread": {"value": single, "unit": UNIT, "cores": 1,
                              "sample": f"one FP64 forward+backward at B=1, L={L1}, D={D}, {t1:.1f} s"}}


def run_reference(args):
    """Times the oracle itself on every host core: each step, every thread runs
    one FP64 forward+backward over its own bounded sample of the workload
    (B=1, the workload's D, a shorter L), inputs drawn before the timed steps."""
    from concurrent.futures import ThreadPoolExecutor
    from linear_recurrence_sequence_gb300 import synth
    wl = synth.WORKLOADS[args.workload]
    D = wl.D
    cores, model = host_cpu()
    per_step_budget = min(2.0, 150.0 / max(1, args.steps + args.warmup))
    with ThreadPoolExecutor(max_workers=cores) as ex:
        def one_step(samples):
            t0 = time.perf_counter()
            list(ex.map(lambda k: _oracle_fb(*samples[k]), range(cores)))
            return time.perf_counter() - t0
        # calibration: one all-threads step on 256-token samples (the threads
        # share the host's memory system, so a thread runs slower than alone)
        cal = [_oracle_inputs(1, 256, D, 300 + k) for k in range(cores)]
        one_step(cal)
        t_cal = one_step(cal)
        del cal
        L = int(max(64, min(wl.L, 8192, per_step_budget / max(t_cal / 256, 1e-9))))
        L = max(64, (L // 64) * 64)
        samples = [_oracle_inputs(1, L, D, 200 + k) for k in range(cores)]
        for _ in range(args.warmup):
            one_step(samples)
        times = [one_step(samples) for _ in range(args.steps)]
    total = sum(times)
    value = args.steps * cores * L / total / 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"samu_fb_B{wl.B}_L{wl.L}_D{wl.D}", "B": wl.B, "L": wl.L, "D": wl.D,
                   "sample_per_step": f"{cores} x (B=1, L={L}, D={D})",
                   "sample_note": f"the sample's L is shorter than the workload's L={wl.L} so that the run "
                                  "ends within a few minutes: the oracle is one sequential pass over the "
                                  "tokens, so its tokens per second do not depend on L"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "cpu_model": model,
                         "sample": f"each step {cores} threads, each one FP64 forward+backward over its own "
                                   f"B=1, L={L}, D={D} sample"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
def run_ours(args, rank, world, local):
    import numpy as np
    import torch
    import torch.distributed as dist
    from linear_recurrence_sequence_gb300 import api, synth

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = synth.WORKLOADS[args.workload]
    if wl.kind != "samu":
        raise SystemExit("bench.py times the SAMU mixer workloads")
    B, L, D = wl.B, wl.L, wl.D
    M = D // 2
    BLD = B * L * D
    inp = wl.make(shard_seed(wl.seeds[0], rank))
    t = api.samu_tensors_from_numpy(inp, dev)
    nsaved, nscratch = api.samu_workspace_bytes(B, L, D)
    saved = torch.empty(nsaved, dtype=torch.uint8, device=dev)
    scratch = torch.empty(nscratch, dtype=torch.uint8, device=dev)
    fo = {"y": torch.empty((B, L, D), dtype=torch.bfloat16, device=dev),
          "hT": torch.empty((B, M, 2), dtype=torch.float32, device=dev)}
    go = {"dx_sel": torch.empty((B, L, D), dtype=torch.bfloat16, device=dev),
          "dw": torch.empty((B, L, D), dtype=torch.bfloat16, device=dev),
          "dh0": torch.empty((B, M, 2), dtype=torch.float32, device=dev),
          "dnu": torch.empty((M,), dtype=torch.float32, device=dev),
          "dtheta": torch.empty((M,), dtype=torch.float32, device=dev),
          "dw_phi": torch.empty((D + 1,), dtype=torch.float32, device=dev),
          "dw_r": torch.empty((D + 1,), dtype=torch.float32, device=dev),
          "da_phi": torch.empty((1,), dtype=torch.float32, device=dev),
          "da_r": torch.empty((1,), dtype=torch.float32, device=dev)}

    def step(x_sel, w, dy):
        api.samu_forward(x_sel, w, t["h0"], t["reset"], t["nu"], t["theta"], t["w_phi"], t["w_r"],
                         t["a_phi"], t["a_r"], out=fo, saved=saved, scratch=scratch)
        return api.samu_backward(dy, t["dhT"], x_sel, w, t["h0"], t["reset"], t["nu"], t["theta"],
                                 t["w_phi"], t["w_r"], t["a_phi"], t["a_r"], saved, out=go,
                                 scratch=scratch)

    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        flush.zero_()
        step(t["x_sel"], t["w"], t["dy"])
    torch.cuda.synchronize(dev)
    if api.device_status(scratch) != 0:
        raise RuntimeError("device-side wait timed out during warm-up")

    # The step as one CUDA graph (the same launches, without the per-call host
    # work); captured on a side stream after the eager warm-up.
    cap_stream = torch.cuda.Stream(dev)
    cap_stream.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(cap_stream):
        step(t["x_sel"], t["w"], t["dy"])
    torch.cuda.current_stream(dev).wait_stream(cap_stream)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap_stream):
        step(t["x_sel"], t["w"], t["dy"])
    # untimed replays until the GPU has been busy for WARM_S seconds (clocks and
    # memory settle; a short --warmup alone can leave the first timed steps slow)
    n_warm = 0
    t_warm = time.perf_counter()
    while n_warm < 3 or time.perf_counter() - t_warm < WARM_S:
        for _ in range(8):
            flush.zero_()
            graph.replay()
        n_warm += 8
        torch.cuda.synchronize(dev)

    K = args.steps
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    sampler = ClockSampler(gpu_selector(dev))
    sampler.start()
    time.sleep(0.1)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    for i in range(K):
        flush.zero_()
        ev0[i].record()
        graph.replay()
        ev1[i].record()
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    if api.device_status(scratch) != 0:
        raise RuntimeError("device-side wait timed out during the timed region")
    step_ms = [ev0[i].elapsed_time(ev1[i]) for i in range(K)]
    total_ms = reduce_max(sum(step_ms), world, dev)
    ms_per_step = total_ms / K
    value = world * B * L * K / (total_ms / 1e3) / 1e6

    # Per-kernel durations: the same steps again, eagerly, with the library's
    # own CUDA events around every launch (on the launching stream; this
    # serialises the launches, so these steps are not part of the value).
    KP = max(3, min(K, 20))
    cap = KP * 8
    api.profile_begin(cap)
    for i in range(KP):
        flush.zero_()
        step(t["x_sel"], t["w"], t["dy"])
    torch.cuda.synchronize(dev)
    records, n_launch_records = api.profile_end(cap)
    if api.device_status(scratch) != 0:
        raise RuntimeError("device-side wait timed out during the per-kernel pass")

    # per-kernel averages and the dominant kernel's roofline
    per = {}
    launches_prof = 0
    for name, ms in records:
        per.setdefault(name, []).append(ms)
        launches_prof += LAUNCHES_PER_RECORD.get(name, 1)
    launches = launches_prof // KP * K   # the timed steps launch the same kernels
    avg = {k: sum(v) / len(v) for k, v in per.items()}
    dom = max((k for k in avg if k in KERNEL_BYTES_PER_BLD), key=lambda k: avg[k] * len(per[k]))
    peak, peak_src = load_peak()
    alg = KERNEL_BYTES_PER_BLD[dom] * BLD
    achieved = alg / (avg[dom] / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                else "fallback 6.8 TB/s", "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": load_traffic(dom, BLD), "algorithmic_bytes": alg,
                "avg_launch_ms": round(avg[dom], 5), "timing": f"library CUDA events, {KP} eager steps"}

    # end to end through the public API with pinned host buffers: every step
    # copies its inputs in (pinned host -> device) and its results out
    # (device -> pinned host) inside the timed region.  Two buffer sets and two
    # copy streams let step i+1's inputs and step i-1's results move while
    # step i computes, as a training input pipeline would.
    K2 = args.e2e_steps if args.e2e_steps is not None else max(10, min(K, 50))   # pipeline fill amortised
    hin = [t[k].cpu().pin_memory() for k in ("x_sel", "w", "dy")]
    small_keys = ("dh0", "dnu", "dtheta", "dw_phi", "dw_r", "da_phi", "da_r")
    sets = []
    for _ in range(2):
        dfo = {"y": torch.empty((B, L, D), dtype=torch.bfloat16, device=dev),
               "hT": torch.empty((B, M, 2), dtype=torch.float32, device=dev)}
        dgo = {"dx_sel": torch.empty((B, L, D), dtype=torch.bfloat16, device=dev),
               "dw": torch.empty((B, L, D), dtype=torch.bfloat16, device=dev),
               "dh0": torch.empty((B, M, 2), dtype=torch.float32, device=dev),
               "dnu": torch.empty((M,), dtype=torch.float32, device=dev),
               "dtheta": torch.empty((M,), dtype=torch.float32, device=dev),
               "dw_phi": torch.empty((D + 1,), dtype=torch.float32, device=dev),
               "dw_r": torch.empty((D + 1,), dtype=torch.float32, device=dev),
               "da_phi": torch.empty((1,), dtype=torch.float32, device=dev),
               "da_r": torch.empty((1,), dtype=torch.float32, device=dev)}
        sets.append({
            "din": [torch.empty_like(t["x_sel"]) for _ in range(3)],
            "fo": dfo, "go": dgo,
            "hout": [torch.empty((B, L, D), dtype=torch.bfloat16).pin_memory() for _ in range(3)],
            "hsmall": {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in dgo.items()
                       if k in small_keys},
            "in_ready": torch.cuda.Event(), "done": torch.cuda.Event(), "out_read": torch.cuda.Event(),
        })
    h2d = 3 * BLD * 2
    d2h = 3 * BLD * 2 + 4 * (B * M * 2)
    copy_ev = []   # per timed step: (H2D start, H2D end, D2H start, D2H end) events
    comp = torch.cuda.current_stream(dev)
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)

    def e2e_steps(n, timed=False):
        for i in range(n):
            S = sets[i % 2]
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)] if timed else None
            with torch.cuda.stream(s_in):
                s_in.wait_event(S["done"])            # step i-2 has finished with this set's inputs
                if timed:
                    ev[0].record(s_in)
                for d_, h_ in zip(S["din"], hin):
                    d_.copy_(h_, non_blocking=True)
                if timed:
                    ev[1].record(s_in)
                S["in_ready"].record(s_in)
            comp.wait_event(S["in_ready"])
            comp.wait_event(S["out_read"])           # step i-2's results have left this set
            go_i = S["go"]
            fo_i = S["fo"]
            api.samu_forward(S["din"][0], S["din"][1], t["h0"], t["reset"], t["nu"], t["theta"], t["w_phi"],
                             t["w_r"], t["a_phi"], t["a_r"], out=fo_i, saved=saved, scratch=scratch)
            g = api.samu_backward(S["din"][2], t["dhT"], S["din"][0], S["din"][1], t["h0"], t["reset"], t["nu"],
                                  t["theta"], t["w_phi"], t["w_r"], t["a_phi"], t["a_r"], saved, out=go_i,
                                  scratch=scratch)
            S["done"].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(S["done"])
                if timed:
                    ev[2].record(s_out)
                for h_, d_ in zip(S["hout"], (fo_i["y"], g["dx_sel"], g["dw"])):
                    h_.copy_(d_, non_blocking=True)
                for k in small_keys:
                    S["hsmall"][k].copy_(g[k], non_blocking=True)
                if timed:
                    ev[3].record(s_out)
                S["out_read"].record(s_out)
            if timed:
                copy_ev.append(ev)

    for S in sets:   # events start "recorded" so that the first waits pass
        S["done"].record(comp)
        S["out_read"].record(comp)
    e2e_steps(2)     # pins and warms the copy path
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    e2e_steps(K2, timed=True)
    comp.wait_stream(s_out)
    comp.wait_stream(s_in)
    e1.record(comp)
    e1.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    d2h += sum(v.numel() * 4 for k, v in sets[0]["hsmall"].items() if k != "dh0")
    # copy rates inside the timed region: each step's H2D (resp. D2H) block
    # between its own events on the copy stream
    h2d_ms = statistics.median(ev[0].elapsed_time(ev[1]) for ev in copy_ev)
    d2h_ms = statistics.median(ev[2].elapsed_time(ev[3]) for ev in copy_ev)
    # share of the timed region during which each copy direction was busy
    # (both near 1: the two directions ran side by side the whole time)
    h2d_busy = sum(ev[0].elapsed_time(ev[1]) for ev in copy_ev) / e2e_ms
    d2h_busy = sum(ev[2].elapsed_time(ev[3]) for ev in copy_ev) / e2e_ms
    e2e_ms = reduce_max(e2e_ms, world, dev)
    e2e_value = world * B * L * K2 / (e2e_ms / 1e3) / 1e6

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "io_dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"samu_fb_B{B}_L{L}_D{D}", "B": B, "L": L, "D": D, "grad_dtype": "bf16",
                   "h0": wl.h0, "reset_p": wl.reset_p, "seed": shard_seed(wl.seeds[0], rank),
                   "l2": "flushed before every timed step (256 MiB memset outside the step events)",
                   "launch": "the step (forward + backward through the C ABI) replayed as one CUDA graph",
                   "warmup_replays": n_warm,
                   "per_gpu_batch": B, "item_transition": args.transition},
        "achieved_step_gbs": round(STEP_BYTES_PER_BLD * BLD / (ms_per_step / 1e3) / 1e9, 1),
        "roofline": roofline,
        "kernels_avg_ms": {k: round(v, 5) for k, v in sorted(avg.items())},
        "gpu_launches": launches,
        "e2e": {"value": round(e2e_value, 3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": K2, "ms_per_step": round(e2e_ms / K2, 4),
                "h2d_gbs": round(h2d / (h2d_ms / 1e3) / 1e9, 1), "d2h_gbs": round(d2h / (d2h_ms / 1e3) / 1e9, 1),
                "h2d_busy": round(h2d_busy, 3), "d2h_busy": round(d2h_busy, 3),
                "overlap": "two buffer sets; H2D of step i+1 and D2H of step i-1 overlap step i",
                "rates": "median per-step H2D and D2H block durations between events on the copy streams; "
                         "*_busy: their summed durations over the timed region"},
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(D)
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# --sweep: every workload family, F+B replayed as a CUDA graph (L2 flushed
# before every step), per-kernel durations from an eager pass with the
# library's events, achieved bytes against the algorithmic minimum
# (SAMU 16 B*L*D, RG-LRU 22 B*L*D with BF16 gradients).  One JSON line each.
SWEEP_BYTES_PER_BLD = {"samu": 16.0, "rglru": 22.0, "rglru_proj": 10.0}


def workload_step(wl, dev):
    """One forward+backward of workload `wl` through the C ABI on resident
    inputs and preallocated outputs (BF16 gradients); returns (step, scratch)."""
    import torch
    from linear_recurrence_sequence_gb300 import api
    B, L, D = wl.B, wl.L, wl.D
    inp = wl.make()
    bf, f32 = torch.bfloat16, torch.float32
    if wl.kind == "samu":
        M = D // 2
        t = api.samu_tensors_from_numpy(inp, dev)
        nsaved, nscratch = api.samu_workspace_bytes(B, L, D)
        fo = {"y": torch.empty((B, L, D), dtype=bf, device=dev), "hT": torch.empty((B, M, 2), dtype=f32, device=dev)}
        go = {"dx_sel": torch.empty((B, L, D), dtype=bf, device=dev), "dw": torch.empty((B, L, D), dtype=bf, device=dev),
              "dh0": torch.empty((B, M, 2), dtype=f32, device=dev), "dnu": torch.empty((M,), dtype=f32, device=dev),
              "dtheta": torch.empty((M,), dtype=f32, device=dev), "dw_phi": torch.empty((D + 1,), dtype=f32, device=dev),
              "dw_r": torch.empty((D + 1,), dtype=f32, device=dev), "da_phi": torch.empty((1,), dtype=f32, device=dev),
              "da_r": torch.empty((1,), dtype=f32, device=dev)}
    elif wl.kind == "rglru_proj":
        t = api.rglru_proj_tensors_from_numpy(inp, dev)
        nsaved, nscratch = api.rglru_proj_workspace_bytes(B, L, D)
        dk = D // api.PROJ_BLOCKS
        fo = {"y": torch.empty((B, L, D), dtype=bf, device=dev), "hT": torch.empty((B, D), dtype=f32, device=dev)}
        go = {"dx": torch.empty((B, L, D), dtype=bf, device=dev),
              "dw_x": torch.empty((api.PROJ_BLOCKS, dk, dk), dtype=f32, device=dev),
              "dw_a": torch.empty((api.PROJ_BLOCKS, dk, dk), dtype=f32, device=dev),
              "db_x": torch.empty((D,), dtype=f32, device=dev), "db_a": torch.empty((D,), dtype=f32, device=dev),
              "dalpha": torch.empty((D,), dtype=f32, device=dev), "dh0": torch.empty((B, D), dtype=f32, device=dev)}
    else:
        t = api.rglru_tensors_from_numpy(inp, dev)
        nsaved, nscratch = api.rglru_workspace_bytes(B, L, D)
        fo = {"y": torch.empty((B, L, D), dtype=bf, device=dev), "hT": torch.empty((B, D), dtype=f32, device=dev)}
        go = {"dx": torch.empty((B, L, D), dtype=bf, device=dev), "dlx": torch.empty((B, L, D), dtype=bf, device=dev),
              "dla": torch.empty((B, L, D), dtype=bf, device=dev), "dalpha": torch.empty((D,), dtype=f32, device=dev),
              "dh0": torch.empty((B, D), dtype=f32, device=dev)}
    saved = torch.empty(nsaved, dtype=torch.uint8, device=dev)
    scratch = torch.empty(nscratch, dtype=torch.uint8, device=dev)

    def step():
        if wl.kind == "samu":
            api.samu_forward(t["x_sel"], t["w"], t["h0"], t["reset"], t["nu"], t["theta"], t["w_phi"], t["w_r"],
                             t["a_phi"], t["a_r"], out=fo, saved=saved, scratch=scratch)
            api.samu_backward(t["dy"], t["dhT"], t["x_sel"], t["w"], t["h0"], t["reset"], t["nu"], t["theta"],
                              t["w_phi"], t["w_r"], t["a_phi"], t["a_r"], saved, out=go, scratch=scratch)
        elif wl.kind == "rglru_proj":
            p = (t["x"], t["w_x"], t["b_x"], t["w_a"], t["b_a"], t["alpha"], t["h0"], t["reset"])
            api.rglru_proj_forward(*p, out=fo, saved=saved, scratch=scratch)
            api.rglru_proj_backward(t["dy"], t["dhT"], *p, saved, out=go, scratch=scratch)
        else:
            api.rglru_forward(t["x"], t["lx"], t["la"], t["alpha"], t["h0"], t["reset"], out=fo, saved=saved,
                              scratch=scratch)
            api.rglru_backward(t["dy"], t["dhT"], t["x"], t["lx"], t["la"], t["alpha"], t["h0"], t["reset"], saved,
                               out=go, scratch=scratch)

    return step, scratch


def sweep_one(name, dev, K, W, transition):
    import torch
    from linear_recurrence_sequence_gb300 import api, synth
    wl = synth.WORKLOADS[name]
    B, L, D = wl.B, wl.L, wl.D
    step, scratch = workload_step(wl, dev)

    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(W):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    cs = torch.cuda.Stream(dev)
    cs.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(cs):
        step()
    torch.cuda.current_stream(dev).wait_stream(cs)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cs):
        step()
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for i in range(K):
        flush.zero_()
        ev0[i].record()
        graph.replay()
        ev1[i].record()
    torch.cuda.synchronize(dev)
    if api.device_status(scratch) != 0:
        raise RuntimeError(f"device-side wait timed out ({name})")
    ms = sorted(ev0[i].elapsed_time(ev1[i]) for i in range(K))
    ms_mean = sum(ms) / K
    KP = max(3, min(K, 10))
    api.profile_begin(KP * 10)
    for _ in range(KP):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    records, _ = api.profile_end(KP * 10)
    per = {}
    for kname, kms in records:
        per.setdefault(kname, []).append(kms)
    BLD = B * L * D
    peak, _ = load_peak()
    alg = SWEEP_BYTES_PER_BLD[wl.kind] * BLD
    gbs = alg / (ms_mean / 1e3) / 1e9
    return {"workload": name, "kind": wl.kind, "B": B, "L": L, "D": D, "steps": K,
            "item_transition": transition if wl.kind == "samu" else None,
            "ms_per_step": round(ms_mean, 5), "ms_min": round(ms[0], 5), "ms_max": round(ms[-1], 5),
            "Mtok_per_s": round(B * L / (ms_mean / 1e3) / 1e6, 3),
            "algorithmic_bytes": alg, "achieved_gbs": round(gbs, 1), "frac_of_measured_peak": round(gbs / peak, 4),
            "frac_of_8tbs": round(gbs / 8000.0, 4),
            "kernels_avg_ms": {k: round(sum(v) / len(v), 5) for k, v in sorted(per.items())}}


# Decode step (one token of each of B sequences): 14 B*D bytes per step
# (x_sel, w, y in BF16; the FP32 state read and written).
DECODE_WORKLOADS = {"decode_B256_D2048": (256, 2048), "decode_B4096_D2048": (4096, 2048),
                    "decode_B16384_D1024": (16384, 1024)}


def sweep_decode(name, dev, K, W):
    import torch
    from linear_recurrence_sequence_gb300 import api, synth
    B, D = DECODE_WORKLOADS[name]
    M = D // 2
    inp = synth.samu_inputs(B, 1, D, 0, h0=True, reset_p=0.0)
    t = api.samu_tensors_from_numpy(inp, dev)
    x, w = t["x_sel"][:, 0].contiguous(), t["w"][:, 0].contiguous()
    params = api.samu_decode_prepare(t["nu"], t["theta"], t["w_phi"], t["w_r"], t["a_phi"], t["a_r"])
    state = t["h0"].clone()
    out = {"y": torch.empty((B, D), dtype=torch.bfloat16, device=dev)}

    def step():
        api.samu_decode_step(x, w, state, params, None, out=out)

    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(W):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    cs = torch.cuda.Stream(dev)
    cs.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(cs):
        step()
    torch.cuda.current_stream(dev).wait_stream(cs)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cs):
        step()
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for i in range(K):
        flush.zero_()
        ev0[i].record()
        graph.replay()
        ev1[i].record()
    torch.cuda.synchronize(dev)
    ms = sorted(ev0[i].elapsed_time(ev1[i]) for i in range(K))
    ms_mean = sum(ms) / K
    KP = max(3, min(K, 10))
    api.profile_begin(KP * 2)
    for _ in range(KP):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    records, _ = api.profile_end(KP * 2)
    kms = [r[1] for r in records]
    peak, _ = load_peak()
    alg = 14.0 * B * D
    gbs = alg / (ms_mean / 1e3) / 1e9
    return {"workload": name, "kind": "samu_decode", "B": B, "L": 1, "D": D, "steps": K,
            "ms_per_step": round(ms_mean, 5), "ms_min": round(ms[0], 5), "ms_max": round(ms[-1], 5),
            "Mtok_per_s": round(B / (ms_mean / 1e3) / 1e6, 3),
            "algorithmic_bytes": alg, "achieved_gbs": round(gbs, 1), "frac_of_measured_peak": round(gbs / peak, 4),
            "frac_of_8tbs": round(gbs / 8000.0, 4),
            "kernels_avg_ms": {"samu_decode_step_kernel": round(sum(kms) / max(1, len(kms)), 5)}}


# One RecurrentBlock around the SAMU mixer (widths Dm, D, F = 3 Dm), F+B as a
# CUDA graph after an L2 flush, like the mixer workloads.  The block is
# dominated by its dense contractions: 18 B L Dm (D + F) flops per F+B (the
# forward's 2 B L Dm (3 D + 3 F), and the same again for dX and for dW), so the
# roofline line is the contraction kernel's achieved TFLOP/s (all its launches
# of a step, eager events) against the measured BF16 tensor-core peak.
# Shapes: the mixer's short shape (B4 L4K, both widths 1024); the pages'
# 400M-width block (Dm 1024, recurrent width D 1536) at their ablation batch
# B4 L2K; the 1.3B widths (Dm 2048, D 2560) at the mixer's medium length.
# The RG-LRU block (rglru_block_*: the same layers around the RG-LRU with its
# gate projections) at the same shapes: the pages' single-block comparison.
BLOCK_SHAPES = {"short": (4, 4096, 1024, 1024), "400m": (4, 2048, 1024, 1536), "medium": (1, 8192, 2048, 2560)}
BLOCK_WORKLOADS = {f"{pre}block_{k}": v + (mix,) for pre, mix in (("", "samu"), ("rglru_", "rglru"))
                   for k, v in BLOCK_SHAPES.items()}
MIXER_KERNELS = {"samu": ("samu_ctrl_fwd_kernel", "samu_fwd_maps_kernel", "samu_fwd_replay_kernel",
                          "samu_bwd_maps_kernel", "samu_bwd_main_kernel", "samu_ctrl_bwd_kernel", "samu_params_kernel"),
                 "rglru": ("rglru_scan_fwd_kernel", "rglru_scan_bwd_kernel", "rglru_alpha_kernels",
                           "proj_gemm_kernel<logits>", "proj_gemm_kernel<dx, dW>", "proj_pack_kernel")}


def block_step(B, L, Dm, D, dev, seed=0, mixer="samu"):
    """One block forward+backward through the C ABI on resident inputs and
    preallocated outputs; returns (step, scratch)."""
    import torch
    from linear_recurrence_sequence_gb300 import api, synth
    inp = synth.block_inputs(B, L, Dm, D, seed, h0=False, reset_p=0.0, mixer=mixer)
    t = api.block_tensors_from_numpy(inp, dev)
    nsaved, nscratch = api.samu_block_workspace_bytes(B, L, Dm, D, mixer)
    saved = torch.empty(nsaved, dtype=torch.uint8, device=dev)
    scratch = torch.empty(nscratch, dtype=torch.uint8, device=dev)
    sshape = (B, D // 2, 2) if mixer == "samu" else (B, D)
    fo = {"out": torch.empty((B, L, Dm), dtype=torch.bfloat16, device=dev),
          "hT": torch.empty(sshape, dtype=torch.float32, device=dev)}
    go = None

    def step():
        nonlocal go
        api.samu_block_forward(t["x"], t["params"], t["h0"], t["reset"], out=fo, saved=saved, scratch=scratch)
        go = api.samu_block_backward(t["dout"], t["dhT"], t["x"], t["params"], t["h0"], t["reset"], saved,
                                     out=go, scratch=scratch)

    return step, scratch


def sweep_block(name, dev, K, W):
    import torch
    from linear_recurrence_sequence_gb300 import api
    B, L, Dm, D, mixer = BLOCK_WORKLOADS[name]
    F = 3 * Dm
    step, scratch = block_step(B, L, Dm, D, dev, mixer=mixer)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(W):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    cs = torch.cuda.Stream(dev)
    cs.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(cs):
        step()
    torch.cuda.current_stream(dev).wait_stream(cs)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cs):
        step()
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for i in range(K):
        flush.zero_()
        ev0[i].record()
        graph.replay()
        ev1[i].record()
    torch.cuda.synchronize(dev)
    if api.device_status(scratch) != 0:
        raise RuntimeError(f"device-side wait timed out ({name})")
    ms = sorted(ev0[i].elapsed_time(ev1[i]) for i in range(K))
    ms_mean = sum(ms) / K
    KP = max(3, min(K, 10))
    cap = KP * 64
    api.profile_begin(cap)
    for _ in range(KP):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    records, n = api.profile_end(cap)
    per = {}
    for kname, kms in records:
        per[kname] = per.get(kname, 0.0) + kms / KP    # per step: all launches of the kernel
    flops = 18.0 * B * L * Dm * (D + F)
    gemm_ms = per.get("block_gemm_kernel", float("nan"))
    tflops = flops / (gemm_ms / 1e3) / 1e12
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        peak, peak_src = float(pk["bf16_tflops"]), "measured (bf16_tflops, burst)"
    except Exception:
        peak, peak_src = 1900.0, "fallback"
    mixer_ms = sum(per.get(k, 0.0) for k in MIXER_KERNELS[mixer])
    eager_ms = sum(per.values())
    return {"workload": name, "kind": f"{mixer}_block", "B": B, "L": L, "Dm": Dm, "D": D, "F": F, "steps": K,
            "ms_per_step": round(ms_mean, 5), "ms_min": round(ms[0], 5), "ms_max": round(ms[-1], 5),
            "Mtok_per_s": round(B * L / (ms_mean / 1e3) / 1e6, 3),
            "roofline": {"bound": "tensor", "kernel": "block_gemm_kernel", "flops_per_step": flops,
                         "kernel_ms_per_step": round(gemm_ms, 5), "achieved": round(tflops, 1), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(tflops / peak, 4), "peak_source": peak_src},
            "mixer_share_of_eager_step": round(mixer_ms / eager_ms, 4) if eager_ms > 0 else None,
            "launches_per_step": n // KP,
            "kernels_ms_per_step": {k: round(v, 5) for k, v in sorted(per.items())}}


# ---------------------------------------------------------------------------
# --compare-pages: SAMU vs RG-LRU with its 16-block gate projections, F+B, on
# the pages' comparison shapes, timed the pages' way: two rounds (RG-LRU
# first, then SAMU first), each 3 warm-up and 5 timed samples per mixer;
# every sample is one eager F+B between CUDA events on the stream, after an L2
# flush; the median of the 10 samples with their range and the raw samples.
# The pages' H800 figures: the absolute pair at B1 L8192 D1024 and, for their
# four primary shapes, the time reduction (t_RG - t_SAMU) / t_RG.
PAGES_SHAPES = [
    # (B, L, D, pages SAMU ms, pages RG-LRU ms, pages reduction %)
    (1, 8192, 1024, 1.801, 1.603, None),
    (4, 2048, 2048, None, None, 24.6),
    (1, 8192, 2560, None, None, 27.6),
    (1, 32768, 1024, None, None, 37.3),
    (1, 32768, 2048, None, None, 40.2),
]


# The pages' single-block table: one complete RecurrentBlock, F+B, SAMU
# 5.8-7.6 % faster than RG-LRU over its three block shapes (the per-shape
# values are not printed).
PAGES_BLOCK_REDUCTION = "5.8-7.6"


def run_compare(args, local):
    import statistics
    import torch
    from linear_recurrence_sequence_gb300 import synth
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for (B, L, D, p_samu, p_rg, p_red) in PAGES_SHAPES:
        wls = {"samu": synth.Workload(f"samu_B{B}_L{L}_D{D}", "samu", B, L, D, (0,), h0=False),
               "rglru_proj": synth.Workload(f"rglru_proj_B{B}_L{L}_D{D}", "rglru_proj", B, L, D, (0,), h0=False)}
        steps = {k: workload_step(wl, dev)[0] for k, wl in wls.items()}
        samples = {k: [] for k in wls}

        def measure(kind):
            for _ in range(3):
                flush.zero_()
                steps[kind]()
            for _ in range(5):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                steps[kind]()
                e1.record()
                e1.synchronize()
                samples[kind].append(e0.elapsed_time(e1))

        for order in (("rglru_proj", "samu"), ("samu", "rglru_proj")):
            for kind in order:
                measure(kind)
        line = {"compare": "pages_shapes", "B": B, "L": L, "D": D,
                "protocol": "2 rounds (RG-LRU first, then SAMU first) x (3 warm-up + 5 samples); eager F+B "
                            "between CUDA events after an L2 flush; median of 10 [min, max]"}
        for kind, pages_ms in (("samu", p_samu), ("rglru_proj", p_rg)):
            v = samples[kind]
            line[kind] = {"median_ms": round(statistics.median(v), 5), "min_ms": round(min(v), 5),
                          "max_ms": round(max(v), 5), "samples_ms": [round(x, 5) for x in v],
                          "pages_h800_ms": pages_ms}
        sm, rm = line["samu"]["median_ms"], line["rglru_proj"]["median_ms"]
        line["samu_time_reduction_percent"] = round(100.0 * (rm - sm) / rm, 1)   # (t_RG - t_SAMU) / t_RG
        line["pages_time_reduction_percent"] = (p_red if p_red is not None
                                                else round(100.0 * (p_rg - p_samu) / p_rg, 1))
        print(json.dumps(line), flush=True)
        del steps
        torch.cuda.empty_cache()
    # the single-block table: the same block around each mixer, same protocol
    for name, (B, L, Dm, D) in BLOCK_SHAPES.items():
        steps = {k: block_step(B, L, Dm, D, dev, mixer=k)[0] for k in ("samu", "rglru")}
        samples = {k: [] for k in steps}

        def measure_block(kind):
            for _ in range(3):
                flush.zero_()
                steps[kind]()
            for _ in range(5):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                steps[kind]()
                e1.record()
                e1.synchronize()
                samples[kind].append(e0.elapsed_time(e1))

        for order in (("rglru", "samu"), ("samu", "rglru")):
            for kind in order:
                measure_block(kind)
        line = {"compare": "pages_block", "block": name, "B": B, "L": L, "Dm": Dm, "D": D, "F": 3 * Dm,
                "protocol": "as the mixer rows: 2 rounds x (3 warm-up + 5 samples), eager F+B of one block "
                            "between CUDA events after an L2 flush; median of 10 [min, max]"}
        for kind in ("samu", "rglru"):
            v = samples[kind]
            line[kind + "_block"] = {"median_ms": round(statistics.median(v), 5), "min_ms": round(min(v), 5),
                                     "max_ms": round(max(v), 5), "samples_ms": [round(x, 5) for x in v]}
        sm, rm = line["samu_block"]["median_ms"], line["rglru_block"]["median_ms"]
        line["samu_time_reduction_percent"] = round(100.0 * (rm - sm) / rm, 1)
        line["pages_time_reduction_percent"] = PAGES_BLOCK_REDUCTION
        print(json.dumps(line), flush=True)
        del steps
        torch.cuda.empty_cache()


def run_sweep(args, local):
    import torch
    from linear_recurrence_sequence_gb300 import synth
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    K = max(5, min(args.steps, 50))
    W = max(3, args.warmup)
    names = (args.only.split(",") if args.only
             else list(synth.WORKLOADS) + list(DECODE_WORKLOADS) + list(BLOCK_WORKLOADS))
    for name in names:
        if name in DECODE_WORKLOADS:
            line = sweep_decode(name, dev, K, W)
        elif name in BLOCK_WORKLOADS:
            line = sweep_block(name, dev, K, W)
        else:
            line = sweep_one(name, dev, K, W, args.transition)
        print(json.dumps(line), flush=True)
        torch.cuda.empty_cache()


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.impl == "reference":
        if rank != 0:
            return 0
        run_reference(args)
        return 0
    if args.sweep:
        if rank == 0:
            set_transition(args)
            run_sweep(args, local)
        return 0
    if args.compare_pages:
        if rank == 0:
            set_transition(args)
            run_compare(args, local)
        return 0
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    try:
        set_transition(args)
        run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
