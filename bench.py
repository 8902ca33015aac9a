#!/usr/bin/env python3
"""Benchmark of the fused row-normalisation path on GB300.

One step = one pass of the whole hot path, each op on its full synthetic
workload, all launched through the C ABI (via the Python binding) on one
stream:
  1. RMSNorm f32 [64, 1024]                     (no residual, gemma off)
  2. add + RMSNorm bf16 [8192, 5120], gemma off  (residual updated in place)
  3. add + RMSNorm bf16 [8192, 5120], gemma on   (a second buffer set)
  4. Q/K RMSNorm + NeoX RoPE bf16, Q and K [26598, 24, 128], theta 1e4
  5. LayerNorm + adaLN modulation bf16 [26598, 3072]
  6. add + RMSNorm bf16 [256, 8192]             (largest decode cell)
  7. silu_and_mul bf16 [256, 2 * 24576]         (largest decode cell)
The metric is achieved HBM throughput: algorithmic bytes (each input read
once, each output written once) per second, summed over the step; rows/s and
per-kernel GB/s with their fractions of the HBM peak are reported beside it.
The step's footprint (~1.7 GB) is far larger than the 129 MB L2 and every
large kernel's operands exceed it, so every launch starts from HBM.  The timed
region runs the steps back to back with CUDA events around the region and
around each launch of the dominant kernel (for the roofline); the per-call
breakdown comes from a second pass with events around every call.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
N > 1 runs under torchrun, one rank per GPU, each rank on its own shard (weak
scaling; RoPE positions continue across ranks).  --impl reference times the CPU
oracle (the plain double-precision definition) on the host instead.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "achieved HBM GB/s and % of GB300 peak per fused norm kernel; rows/sec"
NOMINAL_HBM_GBS = 8000.0
L2_BYTES = 129e6
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")
KERNEL_SOURCES = {
    "qk_norm_rope": "normalisation_rope_transformers_gb300/csrc/qk_norm_rope.cu",
    "add_rmsnorm": "normalisation_rope_transformers_gb300/csrc/rmsnorm.cu",
    "rmsnorm": "normalisation_rope_transformers_gb300/csrc/rmsnorm.cu",
    "ln_modulate": "normalisation_rope_transformers_gb300/csrc/ln_modulate.cu",
    "silu_and_mul": "normalisation_rope_transformers_gb300/csrc/silu_and_mul.cu",
}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", "--iters", dest="steps", type=int, default=3000,
                   help="timed steps (--iters is the same flag)")
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-decode-sweep", action="store_true")
    p.add_argument("--no-back-to-back", action="store_true",
                   help="skip the per-call back-to-back times (e.g. for an ncu launch list)")
    p.add_argument("--no-next-rows", action="store_true")
    p.add_argument("--profile", default=None,
                   help="run only the named call of the step or of the next rows (e.g. qk_norm_rope, "
                        "gelu_and_mul) --steps times, "
                        "for ncu; --rows overrides its row/token count; prints no JSON")
    p.add_argument("--rows", type=int, default=None)
    p.add_argument("--config", type=int, choices=sorted(CONFIG_CALLS), default=None,
                   help="time only the calls of one workload: 1 RMSNorm f32 64x1024, "
                        "2 add + RMSNorm bf16 8192x5120 (gemma off and on), 3 Q/K norm + RoPE "
                        "[26598, 24, 128], 4 LayerNorm + modulation [26598, 3072], 5 the decode "
                        "pair [256, 8192] (and the decode sweep); default: all of them")
    p.add_argument("--seed", type=int, default=None,
                   help="seed of every synthetic input (default: each workload's own seed)")
    return p.parse_args()


# The step's calls that belong to each workload (--config).
CONFIG_CALLS = {
    1: ("rmsnorm_f32_64x1024",),
    2: ("add_rmsnorm_bf16_8192x5120_gemma0", "add_rmsnorm_bf16_8192x5120_gemma1"),
    3: ("qk_norm_rope_bf16_26598x24x128",),
    4: ("ln_modulate_bf16_26598x3072",),
    5: ("add_rmsnorm_bf16_256x8192", "silu_and_mul_bf16_256x49152"),
}


def apply_workload_args(args, synth):
    """--seed replaces the seed of every workload's inputs (the tensors keep
    their own substreams); returns the call names --config selects (None: all)."""
    if args.seed is not None:
        for c in (synth.RMSNORM_F32, synth.ADD_RMSNORM, synth.QK_NORM_ROPE, synth.LN_MODULATE,
                  synth.DECODE):
            c["seed"] = int(args.seed)
    return None if args.config is None else CONFIG_CALLS[args.config]


# ---------------------------------------------------------------------------
# Sharding across ranks (one process per GPU).  Every row and every token is
# independent, so ranks need no data exchange: a rank takes its own rows, and
# RoPE takes global positions, so a token shard passes its own slice of them.
# ---------------------------------------------------------------------------
def shard_range(total, world, rank):
    """Contiguous, balanced [lo, hi) of `total` units for `rank` of `world`."""
    base, extra = divmod(total, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def weak_positions_start(tokens_per_rank, rank):
    """First global position of `rank`'s tokens when every rank holds the same
    number of tokens of one longer sequence (weak scaling)."""
    return rank * tokens_per_rank


def max_over_ranks(value, dist, device=None):
    """The maximum of a float over all ranks (the job's time is its slowest rank)."""
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.item()


# ---------------------------------------------------------------------------
# Workload
# ---------------------------------------------------------------------------
class Call:
    """One launch of the step: its inputs, outputs, byte count and row count."""

    def __init__(self, name, kernel, fn, inputs, outputs, nbytes, rows, rows_unit):
        self.name, self.kernel, self.fn = name, kernel, fn
        self.inputs, self.outputs = inputs, outputs  # dicts name -> device tensor
        self.nbytes, self.rows, self.rows_unit = nbytes, rows, rows_unit


def nbytes(*ts):
    return sum(t.numel() * t.element_size() for t in ts if t is not None)


def step_shapes(synth, selected=None):
    """(name, algorithmic bytes, rows, rows unit) of the seven calls of a step
    (those named in `selected`, when given), from the workload constants alone
    (the reference arm reports the same configuration without building device
    buffers)."""
    out = []
    c = synth.RMSNORM_F32
    n = c["rows"] * c["hidden"]
    out.append(("rmsnorm_f32_64x1024", 4 * (2 * n + c["hidden"]), c["rows"], "rows"))
    c = synth.ADD_RMSNORM
    n = c["rows"] * c["hidden"]
    for gemma in (0, 1):
        out.append(("add_rmsnorm_bf16_8192x5120_gemma%d" % gemma, 2 * (4 * n + c["hidden"]),
                    c["rows"], "rows"))
    c = synth.QK_NORM_ROPE
    n = c["tokens"] * (c["hq"] + c["hk"]) * c["head_dim"]
    out.append(("qk_norm_rope_bf16_26598x24x128", 2 * 2 * n + 2 * 4 * c["head_dim"] + 4 * c["tokens"],
                c["tokens"] * (c["hq"] + c["hk"]), "head rows"))
    c = synth.LN_MODULATE
    n = c["rows"] * c["hidden"]
    out.append(("ln_modulate_bf16_26598x3072", 2 * (2 * n + 2 * c["hidden"]), c["rows"], "rows"))
    c = synth.DECODE
    rows, hidden = max(c["rows"]), max(c["hidden"])
    out.append(("add_rmsnorm_bf16_256x8192", 2 * (4 * rows * hidden + hidden), rows, "rows"))
    out.append(("silu_and_mul_bf16_256x49152", 2 * (rows * 6 * hidden + rows * 3 * hidden), rows,
                "rows"))
    return [o for o in out if selected is None or o[0] in selected]


def step_config(shapes, world):
    """The `config` object of the JSON line (both arms)."""
    step_bytes = sum(s[1] for s in shapes)
    return {"workload": "dit_norm_step: " + " + ".join(s[0] for s in shapes),
            "storage": "bf16 (f32 for the 64x1024 RMSNorm)",
            "bytes_per_step": step_bytes,
            "rows_per_step": {s[0]: s[2] for s in shapes},
            "l2": ("no flush: step footprint %.2f GB >> 129 MB L2; each large call's "
                   "operands exceed L2" % (step_bytes / 1e9) if step_bytes > 2 * L2_BYTES else
                   "no flush: step footprint %.1f MB fits in the 129 MB L2, so steps after the "
                   "first run from L2 (decode-latency regime)" % (step_bytes / 1e6)),
            "parallelism": "dp%d (independent row/token shards, no collective)" % world}


def build_step(nr, synth, torch, device, rank, only=None, selected=None):
    """Device buffers and the seven calls of one step for this rank (only the
    calls whose name starts with `only`, or is in `selected`, when given)."""
    bf16, f32 = torch.bfloat16, torch.float32
    calls = []

    def want(name):
        return ((only is None or name.startswith(only))
                and (selected is None or name in selected))

    c = synth.RMSNORM_F32
    if want("rmsnorm_f32_64x1024"):
        x, _, w = synth.rmsnorm_inputs(c["rows"], c["hidden"], c["seed"], f32, residual=False)
        x, w = x.to(device), w.to(device)
        out = torch.empty_like(x)
        calls.append(Call("rmsnorm_f32_64x1024", "rmsnorm",
                          lambda x=x, w=w, out=out, eps=c["eps"]: nr.rmsnorm(x, w, eps=eps, out=out),
                          {"x": x, "w": w}, {"out": out}, nbytes(x, w, out), c["rows"], "rows"))

    c = synth.ADD_RMSNORM
    for gemma in (False, True):
        if not want("add_rmsnorm_bf16_8192x5120_gemma%d" % gemma):
            continue
        x, res, w = synth.rmsnorm_inputs(c["rows"], c["hidden"], c["seed"], bf16)
        x, res, w = x.to(device), res.to(device), w.to(device)
        out = torch.empty_like(x)
        calls.append(Call("add_rmsnorm_bf16_8192x5120_gemma%d" % gemma, "add_rmsnorm",
                          lambda x=x, w=w, res=res, out=out, g=gemma, eps=c["eps"]:
                          nr.rmsnorm(x, w, residual=res, eps=eps, gemma=g, out=out),
                          {"x": x, "w": w, "residual": res}, {"out": out, "residual": res},
                          nbytes(x, w, res) + nbytes(out, res), c["rows"], "rows"))

    c = synth.QK_NORM_ROPE
    if want("qk_norm_rope_bf16_26598x24x128"):
        q, k, wq, wk, pos = synth.qk_inputs(c["tokens"], c["hq"], c["hk"], c["head_dim"],
                                            c["seed"], bf16, f32,
                                            pos_start=weak_positions_start(c["tokens"], rank))
        q, k, wq, wk, pos = (t.to(device) for t in (q, k, wq, wk, pos))
        qo, ko = torch.empty_like(q), torch.empty_like(k)
        calls.append(Call("qk_norm_rope_bf16_26598x24x128", "qk_norm_rope",
                          lambda q=q, k=k, wq=wq, wk=wk, pos=pos, qo=qo, ko=ko, eps=c["eps"],
                          theta=c["theta"]: nr.qk_norm_rope(q, k, wq, wk, pos, eps=eps,
                                                            theta=theta, q_out=qo, k_out=ko),
                          {"q": q, "k": k, "wq": wq, "wk": wk, "positions": pos},
                          {"q_out": qo, "k_out": ko}, nbytes(q, k, wq, wk, pos, qo, ko),
                          c["tokens"] * (c["hq"] + c["hk"]), "head rows"))

    c = synth.LN_MODULATE
    if want("ln_modulate_bf16_26598x3072"):
        x, sh, sc = synth.ln_inputs(c["rows"], c["hidden"], c["seed"], bf16)
        x, sh, sc = x.to(device), sh.to(device), sc.to(device)
        out = torch.empty_like(x)
        calls.append(Call("ln_modulate_bf16_26598x3072", "ln_modulate",
                          lambda x=x, sh=sh, sc=sc, out=out, eps=c["eps"]:
                          nr.ln_modulate(x, sh, sc, eps=eps, out=out),
                          {"x": x, "shift": sh, "scale": sc}, {"out": out},
                          nbytes(x, sh, sc, out), c["rows"], "rows"))

    c = synth.DECODE
    rows, hidden = max(c["rows"]), max(c["hidden"])
    if want("add_rmsnorm_bf16_256x8192"):
        x, res, w = synth.rmsnorm_inputs(rows, hidden, c["seed"], bf16)
        x, res, w = x.to(device), res.to(device), w.to(device)
        out = torch.empty_like(x)
        calls.append(Call("add_rmsnorm_bf16_256x8192", "add_rmsnorm",
                          lambda x=x, w=w, res=res, out=out, eps=c["eps"]:
                          nr.rmsnorm(x, w, residual=res, eps=eps, out=out),
                          {"x": x, "w": w, "residual": res}, {"out": out, "residual": res},
                          nbytes(x, w, res) + nbytes(out, res), rows, "rows"))
    if want("silu_and_mul_bf16_256x49152"):
        g = synth.silu_inputs(rows, 3 * hidden, c["seed"], bf16).to(device)
        out = torch.empty((rows, 3 * hidden), dtype=bf16, device=device)
        calls.append(Call("silu_and_mul_bf16_256x49152", "silu_and_mul",
                          lambda g=g, out=out: nr.silu_and_mul(g, out=out), {"x": g},
                          {"out": out}, nbytes(g, out), rows, "rows"))
    return calls


# ---------------------------------------------------------------------------
# Clocks during the timed region
# ---------------------------------------------------------------------------
CLOCK_FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
                "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
                "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]


class ClockSampler:
    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.lines = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_id), "--query-gpu=" + ",".join(CLOCK_FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        return time.time()

    def sample_once(self):
        """One synchronous query (read-only), kept with the streamed samples:
        taken right before and right after the timed region, so that a timed
        region shorter than the streaming period still has a clock record."""
        try:
            r = subprocess.run(["nvidia-smi", "-i", str(self.gpu_id),
                                "--query-gpu=" + ",".join(CLOCK_FIELDS),
                                "--format=csv,noheader,nounits"],
                               capture_output=True, text=True, timeout=10)
        except (OSError, subprocess.TimeoutExpired):
            return
        for line in r.stdout.splitlines():
            if line.strip():
                self.lines.append((time.time(), line.strip()))

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if not (t0 <= ts <= t1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(CLOCK_FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_id_for(torch, device):
    try:
        u = torch.cuda.get_device_properties(device).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[device.index or 0] if vis else str(device.index or 0)


# ---------------------------------------------------------------------------
# Peaks and ncu traffic
# ---------------------------------------------------------------------------
def hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def source_hash(rel):
    h = hashlib.sha256()
    for path in (rel, "normalisation_rope_transformers_gb300/csrc/nr_common.cuh"):
        with open(os.path.join(ROOT, path), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def copy_reference(torch, device, nbytes):
    """GB/s of a device-to-device tensor copy moving `nbytes` in total (half
    read, half written), the size of one launch of the dominant kernel: how
    fast plain streaming runs at that size (a copy's start-up and drain weigh
    more on a smaller transfer than on the peak measurement's)."""
    n = max(1, nbytes // 4)  # bf16 elements per buffer
    sets = max(2, (400 * 10 ** 6) // (4 * n) + 1)  # rotate so a buffer is never L2-warm
    src = [torch.empty(n, dtype=torch.bfloat16, device=device).fill_(1.0) for _ in range(sets)]
    dst = [torch.empty_like(src[0]) for _ in range(sets)]
    for i in range(4):
        dst[i % sets].copy_(src[i % sets])
    iters = 40
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for i in range(iters):
        dst[i % sets].copy_(src[i % sets])
    e.record()
    torch.cuda.synchronize(device)
    ms = s.elapsed_time(e) / iters
    return round(4 * n / (ms * 1e-3) / 1e9, 1)


def ncu_traffic(kernel, units):
    """DRAM bytes per launch of `kernel` from the committed ncu capture, scaled
    by the units processed when the capture ran a smaller case (reads grow in
    proportion; writes still dirty in L2 at the kernel's end are written back
    after it and are not counted); None if the kernel's source changed since."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)[kernel]
    except (OSError, KeyError, ValueError):
        return None
    if rec.get("source_hash") != source_hash(KERNEL_SOURCES[kernel]):
        return None
    f = units / rec["units"]
    return {"traffic": int(rec["dram_bytes_per_launch"] * f),
            "traffic_read": int(rec["dram_bytes_read"] * f),
            "traffic_write": int(rec["dram_bytes_write"] * f),
            "traffic_source": "ncu capture of %s, scaled by %s" % (rec["case"], rec["unit"])}


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------
def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)

    import normalisation_rope_transformers_gb300 as nr
    import synth

    selected = apply_workload_args(args, synth)
    calls = build_step(nr, synth, torch, device, rank, selected=selected)
    step_bytes = sum(c.nbytes for c in calls)
    assert [(c.name, c.nbytes, c.rows) for c in calls] == \
        [s[:3] for s in step_shapes(synth, selected)], \
        "step buffers disagree with the workload constants"
    stream = torch.cuda.current_stream(device)

    def step():
        for c in calls:
            c.fn()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(device)

    def per_call_samples(steps):
        """Device time of each call in each of `steps` steps (ms), from CUDA
        events recorded on the launching stream around every call."""
        ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in calls] for _ in range(steps)]
        for i in range(steps):
            for j, c in enumerate(calls):
                ev[i][j][0].record(stream)
                c.fn()
                ev[i][j][1].record(stream)
        torch.cuda.synchronize(device)
        return [[ev[i][j][0].elapsed_time(ev[i][j][1]) for i in range(steps)]
                for j in range(len(calls))]

    # Warm-up (untimed), then a short calibration pass with per-call events:
    # the dominant call (largest median device time) is the one the timed
    # region brackets for the roofline.
    W = max(args.warmup, 3)
    for _ in range(W):
        step()
    calib = [statistics.median(v) for v in per_call_samples(5)]
    dom = max(range(len(calls)), key=lambda j: calib[j])
    barrier()

    # Timed region: K steps; CUDA events bracket the whole region and each
    # launch of the dominant call (no events around the other calls, so the
    # step is timed as it runs back to back).
    K = args.steps
    dom_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for a, b in dom_ev:  # create the CUDA events now, outside the timed region
        a.record(stream)
        b.record(stream)
    barrier()
    sampler = ClockSampler(gpu_id_for(torch, device))
    with sampler:
        t_clock0 = time.time()
        sampler.sample_once()
        barrier()
        t_wall0 = time.time()
        start.record(stream)
        for i in range(K):
            for j, c in enumerate(calls):
                if j == dom:
                    dom_ev[i][0].record(stream)
                    c.fn()
                    dom_ev[i][1].record(stream)
                else:
                    c.fn()
        end.record(stream)
        barrier()
        t_wall1 = time.time()
        sampler.sample_once()
        t_clock1 = time.time()
    # the streamed samples inside the timed region plus the two synchronous
    # samples taken just before and just after it
    clocks = sampler.summary(t_clock0, t_clock1)
    clocks["window"] = "timed region, with one query just before and one just after it"
    elapsed_ms = start.elapsed_time(end)
    dom_samples = [a.elapsed_time(b) for a, b in dom_ev]
    dom_ms = statistics.fmean(dom_samples)
    if world > 1:
        elapsed_ms = max_over_ranks(elapsed_ms, dist, device)

    # Per-call breakdown, after the timed region: events around every call.
    breakdown_steps = min(K, 300)
    samples = per_call_samples(breakdown_steps)
    per_call_ms = [statistics.fmean(v) for v in samples]
    b2b_ms = ({} if args.no_back_to_back else
              {c.name: back_to_back_ms(torch, c.fn) for c in calls if c.nbytes > 2 * L2_BYTES})

    ms_per_step = elapsed_ms / K
    value = world * step_bytes * K / (elapsed_ms * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()

    kernels = {}
    for c, ms, v in zip(calls, per_call_ms, samples):
        gbs = c.nbytes / (ms * 1e-3) / 1e9
        kernels[c.name] = {"us": round(ms * 1e3, 2), "us_median": round(statistics.median(v) * 1e3, 2),
                           "us_min": round(min(v) * 1e3, 2), "bytes": c.nbytes, "GB_s": round(gbs, 1),
                           "frac_of_measured": round(gbs / peak, 4),
                           "frac_of_nominal_8TBs": round(gbs / NOMINAL_HBM_GBS, 4),
                           "rows_per_s": round(c.rows / (ms * 1e-3), 1), "rows_unit": c.rows_unit}
        if c.name in b2b_ms:
            gbs_b2b = c.nbytes / (b2b_ms[c.name] * 1e-3) / 1e9
            kernels[c.name].update({"us_b2b": round(b2b_ms[c.name] * 1e3, 2),
                                    "GB_s_b2b": round(gbs_b2b, 1),
                                    "frac_of_measured_b2b": round(gbs_b2b / peak, 4)})
    dc = calls[dom]
    achieved = dc.nbytes / (dom_ms * 1e-3) / 1e9
    traffic = ncu_traffic(dc.kernel, dc.rows)
    copy_gbs = copy_reference(torch, device, dc.nbytes) if rank == 0 else None

    e2e = run_e2e(args, torch, calls, device, world, barrier, step_bytes)

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": max(args.warmup, 3), "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": step_config([(c.name, c.nbytes, c.rows, c.rows_unit) for c in calls], world),
        "roofline": dict({"bound": "hbm", "kernel": dc.name, "achieved": round(achieved, 1),
                          "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                          "frac": round(achieved / peak, 4),
                          "frac_of_nominal_8TBs": round(achieved / NOMINAL_HBM_GBS, 4),
                          "traffic": None, "algorithmic_bytes": dc.nbytes,
                          "duration_us": round(dom_ms * 1e3, 2),
                          "duration_us_median": round(statistics.median(dom_samples) * 1e3, 2),
                          "duration_us_min": round(min(dom_samples) * 1e3, 2),
                          "duration_us_b2b": (round(b2b_ms[dc.name] * 1e3, 2)
                                              if dc.name in b2b_ms else None),
                          "frac_b2b": (round(dc.nbytes / (b2b_ms[dc.name] * 1e-3) / 1e9 / peak, 4)
                                       if dc.name in b2b_ms else None),
                          "copy_same_bytes_GB_s": copy_gbs,
                          "frac_of_copy_same_bytes": (round(achieved / copy_gbs, 4)
                                                      if copy_gbs else None)},
                         **(traffic or {})),
        "kernels": kernels,
        "kernels_timing": ("per-call CUDA events over %d steps after the timed region (the "
                           "timed region brackets only the dominant call); *_b2b: the call "
                           "alone, %d launches back to back between two CUDA events (median "
                           "of %d), as the next rows are timed, for calls whose operands "
                           "exceed twice the L2" % (breakdown_steps, B2B_LAUNCHES, B2B_REPS)),
        "rows_per_s": round(world * sum(c.rows for c in calls) / (ms_per_step * 1e-3), 1),
        "e2e": e2e,
        "gpu_launches": K * len(calls),
        "clocks": clocks,
    }
    if rank == 0 and not args.no_decode_sweep and args.config in (None, 5):
        result["decode_sweep"] = decode_sweep(nr, synth, torch, device)
    if rank == 0 and not args.no_next_rows and args.config is None:
        result["next_rows"] = next_rows(nr, synth, torch, device, peak)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(fraction=0.5, selected=selected)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


def run_e2e(args, torch, calls, device, world, barrier, step_bytes):
    """Same step through the public API with inputs in pinned host memory: each
    step copies every input host->device, runs the seven calls and copies every
    output device->host, all inside the timed region.  Copies in, kernels and
    copies out run on three streams ordered per call by events, so the two copy
    directions overlap each other and the kernels."""
    h_in = [{k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True).copy_(v.cpu())
             for k, v in c.inputs.items()} for c in calls]
    h_out = [{k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in c.outputs.items()}
             for c in calls]
    h2d = sum(nbytes(*d.values()) for d in h_in)
    d2h = sum(nbytes(*d.values()) for d in h_out)
    s_in, s_k, s_out = (torch.cuda.Stream(device) for _ in range(3))
    main = torch.cuda.current_stream(device)

    # ev_out[j]: call j's outputs have been copied out.  The next step's copy
    # into call j's buffers (some are read and written in place) waits for it.
    ev_out = [None] * len(calls)

    def step():
        for j, (c, hi, ho) in enumerate(zip(calls, h_in, h_out)):
            with torch.cuda.stream(s_in):
                if ev_out[j] is not None:
                    s_in.wait_event(ev_out[j])
                for k, v in hi.items():
                    c.inputs[k].copy_(v, non_blocking=True)
            s_k.wait_stream(s_in)
            with torch.cuda.stream(s_k):
                c.fn()
            s_out.wait_stream(s_k)
            with torch.cuda.stream(s_out):
                for k, v in ho.items():
                    v.copy_(c.outputs[k], non_blocking=True)
                ev_out[j] = torch.cuda.Event()
                ev_out[j].record(s_out)

    # The same copies with no kernels (the host link's time for this step's
    # transfers), for context: the end-to-end step cannot be faster.
    def copies_only():
        for c, hi, ho in zip(calls, h_in, h_out):
            with torch.cuda.stream(s_in):
                for k, v in hi.items():
                    c.inputs[k].copy_(v, non_blocking=True)
            with torch.cuda.stream(s_out):
                for k, v in ho.items():
                    v.copy_(c.outputs[k], non_blocking=True)

    def window(fn, streams, steps):
        """ms per step of `steps` back-to-back calls of fn, max over ranks."""
        barrier()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(main)
        for st in streams:
            st.wait_stream(main)
        for _ in range(steps):
            fn()
        for st in streams:
            main.wait_stream(st)
        e.record(main)
        barrier()
        ms = s.elapsed_time(e)
        if world > 1:
            import torch.distributed as dist

            ms = max_over_ranks(ms, dist, device)
        return ms / steps

    step()
    copies_only()
    # The host link is shared with the rest of the machine and its rate can
    # drop for a while, so the two measurements alternate in short windows and
    # each reports its median window.
    n = max(args.e2e_steps, 1)
    windows = 5
    e2e_ms, copy_ms = [], []
    for _ in range(windows):
        e2e_ms.append(window(step, (s_in, s_k, s_out), n))
        copy_ms.append(window(copies_only, (s_in, s_out), n))
    ms = statistics.median(e2e_ms)
    cms = statistics.median(copy_ms)
    return {"value": round(world * step_bytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n * windows,
            "ms_per_step": round(ms, 3),
            "copies_only_ms_per_step": round(cms, 3),
            "frac_of_copies_only": round(cms / ms, 4),
            "windows_ms_per_step": [round(x, 3) for x in e2e_ms],
            "copies_only_windows_ms_per_step": [round(x, 3) for x in copy_ms],
            "note": "pinned host buffers; H2D, kernels and D2H on three streams ordered per call; "
                    "copies_only = the same transfers with no kernels (host-link bound); %d "
                    "alternating windows of %d steps each, medians reported" % (windows, n)}


def next_row_cases(nr, synth, torch, device, rows_override=None):
    """The ops beyond the seven-call step as (name, make) pairs; make() puts
    the operands on the device and returns (fn, bytes per call, rows).
    rows_override shrinks the row count (for ncu captures)."""
    def n_rows(default):
        return default if rows_override is None else rows_override

    def gated():
        # gated residual + LayerNorm + modulation at the DiT shape, one sample
        rows, hidden = n_rows(synth.LN_MODULATE["rows"]), synth.LN_MODULATE["hidden"]
        res = synth.tensor(5, 20, (rows, hidden), torch.bfloat16).to(device)
        y = synth.tensor(5, 21, (rows, hidden), torch.bfloat16).to(device)
        gate, sh, sc = (synth.tensor(5, i, (1, hidden), torch.bfloat16, std=0.1).to(device)
                        for i in (22, 23, 24))
        o = torch.empty_like(res)
        return (lambda: nr.gated_residual_ln_modulate(res, y, gate, sh, sc, out=o),
                nbytes(res, y, gate, sh, sc) + nbytes(res, o), rows)

    def quant():
        # RMSNorm + e4m3 quantisation with the residual add, at the dense shape
        c = synth.ADD_RMSNORM
        rows = n_rows(c["rows"])
        x, res, w = synth.rmsnorm_inputs(rows, c["hidden"], c["seed"], torch.bfloat16)
        x, res, w = x.to(device), res.to(device), w.to(device)
        codes = torch.empty(x.shape, dtype=torch.uint8, device=device)
        return (lambda: nr.rmsnorm_quant_fp8(x, w, 0.02, residual=res, codes=codes),
                nbytes(x, w, res) + nbytes(res, codes), rows)

    def gelu():
        # tanh-GELU gate times up, prefill-sized: 8192 tokens, intermediate 3 * 5120
        rows = n_rows(8192)
        g = synth.silu_inputs(rows, 3 * 5120, 6, torch.bfloat16).to(device)
        o = torch.empty((rows, 3 * 5120), dtype=torch.bfloat16, device=device)
        return lambda: nr.gelu_and_mul(g, out=o), nbytes(g, o), rows

    def rope_variant(**kw):
        # Q/K [26598, 24, 128] bf16 (the Q/K workload's shape) with a RoPE variant
        def make():
            c = synth.QK_NORM_ROPE
            t = n_rows(c["tokens"])
            q, k, wq, wk, pos = synth.qk_inputs(t, c["hq"], c["hk"], c["head_dim"], 7,
                                                torch.bfloat16, torch.float32)
            if kw.get("mrope_sections"):
                # three position rows (t, h, w), as a vision-language model's image tokens
                pos = torch.stack([pos // 1024, (pos // 32) % 32, pos % 32]).to(torch.int32)
            if kw.get("llama3"):
                pos = (pos * 4).to(torch.int32)  # positions up to ~106k
            q, k, wq, wk, pos = (v.to(device) for v in (q, k, wq, wk, pos))
            qo, ko = torch.empty_like(q), torch.empty_like(k)
            nb = nbytes(q, k, wq, wk, pos) + nbytes(qo, ko)
            return (lambda: nr.qk_norm_rope_ex(q, k, wq, wk, pos, q_out=qo, k_out=ko, **kw), nb,
                    t)
        return make

    return [("gated_residual_ln_modulate_bf16_26598x3072", gated),
            ("rmsnorm_quant_fp8_bf16_8192x5120", quant),
            ("gelu_and_mul_bf16_8192x30720", gelu),
            ("qk_norm_rope_mrope_bf16_26598x24x128", rope_variant(
                mrope_sections=(16, 24, 24), theta=1e6)),
            ("qk_norm_rope_gptj_rot64_bf16_26598x24x128", rope_variant(
                rotary_dim=64, interleaved=True)),
            ("qk_norm_rope_llama3_bf16_26598x24x128", rope_variant(
                theta=500000.0, llama3=(8.0, 1.0, 4.0, 8192.0)))]


B2B_LAUNCHES = 20
B2B_REPS = 5


def back_to_back_ms(torch, fn):
    """Device time per launch of `fn` run alone, B2B_LAUNCHES launches back to
    back between two CUDA events (median over B2B_REPS): each launch's start
    overlaps the previous one's drain (programmatic dependent launch), which an
    event recorded between two launches prevents."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    out = []
    for _ in range(B2B_REPS):
        s.record()
        for _ in range(B2B_LAUNCHES):
            fn()
        e.record()
        torch.cuda.synchronize()
        out.append(s.elapsed_time(e) / B2B_LAUNCHES)
    return statistics.median(out)


def next_rows(nr, synth, torch, device, peak):
    """The ops beyond the seven-call step, each timed alone on its own workload
    (mean of CUDA-event times over back-to-back calls, operands larger than L2)."""
    out = {}
    for name, make in next_row_cases(nr, synth, torch, device):
        fn, nb, rows = make()
        iters = 50
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(iters):
            fn()
        e.record()
        torch.cuda.synchronize()
        us = s.elapsed_time(e) * 1e3 / iters
        gbs = nb / (us * 1e-6) / 1e9
        out[name] = {"us": round(us, 2), "bytes": nb, "GB_s": round(gbs, 1),
                     "frac_of_measured": round(gbs / peak, 4),
                     "frac_of_nominal_8TBs": round(gbs / NOMINAL_HBM_GBS, 4),
                     "rows_per_s": round(rows / (us * 1e-6), 1)}
        del fn
    return out


def decode_sweep(nr, synth, torch, device):
    """Latency per call of add+RMSNorm and silu_and_mul over the decode grid,
    both from CUDA graphs of back-to-back calls (so host launch overhead is not
    in the figure): hot = the same buffers every call (L2-warm); cold = the
    calls cycle through enough copies of the buffers to span > 2x the 129 MB
    L2, so every call reads from HBM."""
    c = synth.DECODE
    span = 320 << 20
    out = {}

    def graph_us(fns):
        for f in fns[:3]:
            f()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for f in fns:
                f()
        graph.replay()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        graph.replay()
        e.record()
        torch.cuda.synchronize()
        return s.elapsed_time(e) * 1e3 / len(fns)

    for rows in c["rows"]:
        for hidden in c["hidden"]:
            x, res, w = synth.rmsnorm_inputs(rows, hidden, c["seed"], torch.bfloat16)
            g = synth.silu_inputs(rows, 3 * hidden, c["seed"], torch.bfloat16)
            rms_bytes = nbytes(x, w, res) * 2 - nbytes(w)  # read x, res, w; write out, res
            silu_bytes = nbytes(g) * 3 // 2
            for name, nb in (("add_rmsnorm", rms_bytes), ("silu_and_mul", silu_bytes)):
                sets = int(min(4096, max(2, span // nb)))
                if name == "add_rmsnorm":
                    xs = x.to(device).repeat(sets, 1).view(sets, rows, hidden)
                    rs = res.to(device).repeat(sets, 1).view(sets, rows, hidden)
                    os_ = torch.empty_like(xs)
                    wd = w.to(device)
                    fns = [lambda i=i: nr.rmsnorm(xs[i], wd, residual=rs[i], out=os_[i])
                           for i in range(sets)]
                else:
                    gs = g.to(device).repeat(sets, 1).view(sets, rows, 6 * hidden)
                    os_ = torch.empty((sets, rows, 3 * hidden), dtype=torch.bfloat16,
                                      device=device)
                    fns = [lambda i=i: nr.silu_and_mul(gs[i], out=os_[i]) for i in range(sets)]
                hot_us = graph_us([fns[0]] * 100)
                cold_us = graph_us(fns)
                out["%s_%dx%d" % (name, rows, hidden)] = {
                    "hot_us": round(hot_us, 2), "cold_us": round(cold_us, 2), "bytes": nb,
                    "hot_GB_s": round(nb / (hot_us * 1e-6) / 1e9, 1),
                    "cold_GB_s": round(nb / (cold_us * 1e-6) / 1e9, 1), "cold_sets": sets}
                del fns
    return out


# ---------------------------------------------------------------------------
# CPU oracle (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------
def prepare_oracle_step(fraction, selected=None):
    """Oracle calls over the first `fraction` of each workload's rows (at least
    one row).  The generator is counter-based, so these inputs are exactly the
    leading rows of the full workloads.  Returns [(fn(lo, hi), rows, algorithmic
    bytes)], desc; fn runs the oracle on rows [lo, hi) of its sample."""
    import torch

    import oracle
    import synth

    bf16, f32 = torch.bfloat16, torch.float32
    o = synth.to_oracle
    ops, desc, names = [], [], []

    def rows_of(n):
        return max(1, min(n, int(round(n * fraction))))

    c = synth.RMSNORM_F32
    r = rows_of(c["rows"])
    x, _, w = synth.rmsnorm_inputs(r, c["hidden"], c["seed"], f32, residual=False)
    ops.append((lambda lo, hi, a=o(x), b=o(w): oracle.rmsnorm(a[lo:hi], b), r,
                2 * x.numel() * 4 + w.numel() * 4))
    desc.append("rmsnorm_f32 %d/%d rows" % (r, c["rows"]))
    names.append("rmsnorm_f32_64x1024")
    c = synth.ADD_RMSNORM
    r = rows_of(c["rows"])
    x, res, w = synth.rmsnorm_inputs(r, c["hidden"], c["seed"], bf16)
    for gemma in (False, True):
        ops.append((lambda lo, hi, a=o(x), b=o(w), rr=o(res), g=gemma:
                    oracle.rmsnorm(a[lo:hi], b, residual=rr[lo:hi], gemma=g), r,
                    4 * r * c["hidden"] * 2 + c["hidden"] * 2))
        desc.append("add_rmsnorm gemma%d %d/%d rows" % (gemma, r, c["rows"]))
        names.append("add_rmsnorm_bf16_8192x5120_gemma%d" % gemma)
    c = synth.QK_NORM_ROPE
    t = rows_of(c["tokens"])
    q, k, wq, wk, pos = synth.qk_inputs(t, c["hq"], c["hk"], c["head_dim"], c["seed"], bf16, f32)
    ops.append((lambda lo, hi, a=o(q), b=o(k), wa=o(wq), wb=o(wk), p=pos.numpy(), th=c["theta"]:
                oracle.qk_norm_rope(a[lo:hi], b[lo:hi], wa, wb, p[lo:hi], theta=th), t,
                4 * t * c["hq"] * c["head_dim"] * 2 + t * 4 + 2 * c["head_dim"] * 4))
    desc.append("qk_norm_rope %d/%d tokens" % (t, c["tokens"]))
    names.append("qk_norm_rope_bf16_26598x24x128")
    c = synth.LN_MODULATE
    r = rows_of(c["rows"])
    x, sh, sc = synth.ln_inputs(r, c["hidden"], c["seed"], bf16)
    ops.append((lambda lo, hi, a=o(x), s1=o(sh), s2=o(sc): oracle.ln_modulate(a[lo:hi], s1, s2),
                r, 2 * r * c["hidden"] * 2 + 2 * c["hidden"] * 2))
    desc.append("ln_modulate %d/%d rows" % (r, c["rows"]))
    names.append("ln_modulate_bf16_26598x3072")
    c = synth.DECODE
    rows, hidden = max(c["rows"]), max(c["hidden"])
    r = rows_of(rows)
    x, res, w = synth.rmsnorm_inputs(r, hidden, c["seed"], bf16)
    ops.append((lambda lo, hi, a=o(x), b=o(w), rr=o(res):
                oracle.rmsnorm(a[lo:hi], b, residual=rr[lo:hi]), r, 4 * r * hidden * 2 + hidden * 2))
    desc.append("add_rmsnorm %d/%d rows of 8192" % (r, rows))
    names.append("add_rmsnorm_bf16_256x8192")
    g = synth.silu_inputs(r, 3 * hidden, c["seed"], bf16)
    ops.append((lambda lo, hi, a=o(g): oracle.silu_and_mul(a[lo:hi]), r, 3 * r * 3 * hidden * 2))
    desc.append("silu_and_mul %d/%d rows" % (r, rows))
    names.append("silu_and_mul_bf16_256x49152")
    oracle._load()
    keep = [i for i, n in enumerate(names) if selected is None or n in selected]
    return [ops[i] for i in keep], "; ".join(desc[i] for i in keep)


def oracle_threads():
    """Host threads for the parallel oracle runs: one per core."""
    return max(1, os.cpu_count() or 1)


def time_oracle(ops, threads=1):
    """Wall time of one pass over `ops` and its algorithmic bytes.  With
    threads > 1 each op's rows are split into contiguous chunks run on a thread
    pool (the C oracle releases the GIL while it runs), op after op."""
    secs, nb = 0.0, 0
    if threads <= 1:
        for fn, rows, b in ops:
            t0 = time.perf_counter()
            fn(0, rows)
            secs += time.perf_counter() - t0
            nb += b
        return secs, nb
    from concurrent.futures import ThreadPoolExecutor

    with ThreadPoolExecutor(max_workers=threads) as pool:
        for fn, rows, b in ops:
            n = min(threads, rows)
            bounds = [(i * rows // n, (i + 1) * rows // n) for i in range(n)]
            t0 = time.perf_counter()
            list(pool.map(lambda lh: fn(*lh), bounds))
            secs += time.perf_counter() - t0
            nb += b
    return secs, nb


def cpu_baseline(fraction, selected=None):
    ops, desc = prepare_oracle_step(fraction, selected)
    secs1, nb = time_oracle(ops)
    threads = oracle_threads()
    secs, _ = time_oracle(ops, threads)
    return {"value": round(nb / secs / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": "one pass of the step over %.0f%% of each workload's rows (%s), the C "
                      "oracle in double with each call's rows split over %d host threads, %.1f s; "
                      "single-threaded: %.4f GB/s in %.1f s"
                      % (100 * fraction, desc, threads, secs, nb / secs1 / 1e9, secs1),
            "single_thread_value": round(nb / secs1 / 1e9, 4)}


def run_reference(args):
    """The CPU oracle as the reference arm: each step is the oracle over a
    sample of every workload in the step, sized so the whole run stays within
    about two minutes."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    import synth

    steps, warm = args.steps, max(args.warmup, 3)
    selected = apply_workload_args(args, synth)
    threads = oracle_threads()
    probe_fraction = 1.0 / 256
    ops, _ = prepare_oracle_step(probe_fraction, selected)
    probe_s, _ = time_oracle(ops, threads)
    per_step_budget = min(2.0, 120.0 / (steps + warm))
    fraction = max(1.0 / 26598, min(0.5, probe_fraction * per_step_budget / max(probe_s, 1e-6)))
    ops, desc = prepare_oracle_step(fraction, selected)
    for _ in range(warm):
        time_oracle(ops, threads)
    total_s, total_b = 0.0, 0
    for _ in range(steps):
        s, b = time_oracle(ops, threads)
        total_s += s
        total_b += b
    value = total_b / total_s / 1e9
    sample = ("each step: %s (%.3g of each workload's rows), C oracle with each call's rows "
              "split over %d host threads" % (desc, fraction, threads))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": steps, "warmup": warm,
        "ms_per_step": round(1e3 * total_s / steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": step_config(step_shapes(synth, selected), args.gpus),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def run_profile(args):
    """Run one call of the step (optionally at a smaller row count) --steps
    times after --warmup calls: the target of the ncu captures."""
    import torch

    import normalisation_rope_transformers_gb300 as nr
    import synth

    device = torch.device("cuda", 0)
    apply_workload_args(args, synth)
    if args.rows is not None:
        for cfg, key in ((synth.ADD_RMSNORM, "rows"), (synth.QK_NORM_ROPE, "tokens"),
                         (synth.LN_MODULATE, "rows")):
            cfg[key] = args.rows
    calls = build_step(nr, synth, torch, device, 0, only=args.profile)
    if calls:
        c = calls[0]
        fn, name, nb, rows, unit = c.fn, c.name, c.nbytes, c.rows, c.rows_unit
    else:
        cases = [(n, m) for n, m in next_row_cases(nr, synth, torch, device, args.rows)
                 if n.startswith(args.profile)]
        if not cases:
            raise SystemExit("no call named %s*" % args.profile)
        name = cases[0][0]
        fn, nb, rows = cases[0][1]()
        unit = "rows"
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    for _ in range(args.steps):
        fn()
    torch.cuda.synchronize()
    print("profiled %s x%d (%d bytes per launch, %d %s)" % (name, args.steps, nb, rows, unit))


def main():
    args = parse_args()
    if args.profile:
        run_profile(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
