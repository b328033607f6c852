"""Benchmark of the pi-Attention hot path on one GB300 (or N replicas under torchrun).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C4] [--impl ours|reference]

A step is one pass of the hot path over one batch of synthetic input: the
fused forward (band tiles + skip gather + GQA + epilogue) for the forward
workloads, forward + backward for the training workloads C5 (causal) and C7
(bidirectional).  The default
workload is C4 (B1 H16 Hkv4 N65536 d128 k256 pi1024 S4, bf16), the N=65536
configuration the roofline target is stated for.

Prints one JSON line.  `value` is tokens/s (B*N per step, summed over ranks);
the line also carries useful TFLOP/s (4d FLOPs per attended pair forward, 8d
backward), the roofline of the dominant kernel against the measured peaks in
MEASURED_PEAKS.json, the fp64 oracle timed on this host's cores on a bounded
sample (`cpu_baseline`), an end-to-end number through the public API with
host buffers (`e2e`), the number of kernel launches, and the SM clocks sampled
during the timed region.  `--impl reference` times the oracle instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from structured_sparse_long_gb300.synth import (MODE_ECP, MODE_PI_BIDIR, WORKLOADS, gate_weights,  # noqa: E402
                                                make_inputs)

METRIC = "sparse-attn tokens/s and useful TFLOP/s at N=4K–64K; % of roofline (1×GB300)"
L2_BYTES = 129 * 1024 * 1024
SPIN_CYCLES = 100_000  # device-side spin after each L2 flush (about 50 us at 2 GHz)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
PROFILE_DIR = os.path.join(ROOT, "profiles")


# ----------------------------------------------------------------------------- work accounting

def pairs_per_head(N, k, period, S, mode) -> int:
    """Attended (query, key) pairs of one (b, h), closed forms of the neighbour sets."""
    if mode == MODE_ECP:
        c, total, s = k, 0, 0
        while s * c < N:
            n = min(c, N - s * c)
            total += n * (n + 1) // 2 if s == 0 else n * (c + 1) + n * (n - 1) // 2
            s += 1
        return total
    if mode == MODE_PI_BIDIR:  # |i - j| <= k, and skips on both sides
        kk = min(k, N - 1)
        band = N + 2 * (kk * N - kk * (kk + 1) // 2)
        skip = sum(2 * max(0, N - m * period) for m in range(1, S + 1) if m * period > k)
        return band + skip
    band = N * (k + 1) - k * (k + 1) // 2 if k < N else N * (N + 1) // 2
    skip = sum(max(0, N - m * period) for m in range(1, S + 1) if m * period > k)
    return band + skip


def decode_keys(w) -> int:
    """Neighbours of row N-1 (the decode query): band rows and skip rows N-1 - m*period."""
    i = w.N - 1
    if w.mode == MODE_ECP:
        return i - max(0, (i // w.k_local - 1) * w.k_local) + 1
    band = min(w.k_local, i) + 1
    skip = sum(1 for m in range(1, w.S + 1) if m * w.period > w.k_local and i - m * w.period >= 0)
    return band + skip


def work(w, backward: bool):
    esz = 4 if w.dtype == "f32" else 2
    if w.decode:  # only the neighbour rows of the cache are read
        nk = decode_keys(w)
        pairs = w.B * w.H * nk
        byts = w.B * w.Hkv * nk * w.d * esz * 2 + 2 * w.B * w.H * w.d * esz + 8 * w.B * w.H
        return {"pairs": pairs, "fwd_bytes": byts, "fwd_flops": 4 * w.d * pairs, "bytes": byts,
                "flops": 4 * w.d * pairs}
    pairs = pairs_per_head(w.N, w.k_local, w.period, w.S, w.mode) * w.B * w.H
    qo = w.B * w.H * w.N * w.d * esz
    kv = w.B * w.Hkv * w.N * w.d * esz
    vec = w.B * w.H * w.N * 4
    fwd_bytes = 2 * qo + 2 * kv + vec * (2 if w.mode != MODE_ECP else 1)
    fwd_flops = 4 * w.d * pairs
    res = {"pairs": pairs, "fwd_bytes": fwd_bytes, "fwd_flops": fwd_flops,
           "bytes": fwd_bytes, "flops": fwd_flops}
    if backward:
        bwd_bytes = 4 * qo + 4 * kv + 3 * vec
        res.update(bwd_bytes=bwd_bytes, bwd_flops=8 * w.d * pairs, bwd_flops_10d=10 * w.d * pairs,
                   bytes=fwd_bytes + bwd_bytes, flops=fwd_flops + 8 * w.d * pairs)
    return res


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = {
    "fwd": ("pi_fwd_tc.cu", "pi_common.cuh", "pi_launch.h", "pi_tc_ptx.cuh"),
    "bwd": ("pi_bwd_tc.cu", "pi_common.cuh", "pi_launch.h", "pi_tc_ptx.cuh"),
    "dec": ("pi_decode.cu", "pi_common.cuh", "pi_launch.h", "pi_tc_ptx.cuh"),
}
PROFILE_NAMES = {"fwd": "pi_fwd_tc", "bwd": "pi_bwd_tc", "dec": "pi_decode"}


def _code_only(src: str) -> str:
    """C++/CUDA source without comments and with whitespace runs collapsed: what the compiler sees."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c == '"' or c == "'":  # string or character literal, copied as is
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_sha(kind: str = "fwd") -> str:
    """Hash of the kernel's sources as compiled: comments and layout do not change it."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "structured_sparse_long_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kind: str = "fwd"):
    """DRAM bytes of one forward launch (kind "fwd"), of one backward call, both of its
    kernels (kind "bwd"), or of one decode step (kind "dec"), from a committed ncu summary --
    if it was taken on the current kernel source (else None)."""
    path = os.path.join(PROFILE_DIR, f"{PROFILE_NAMES[kind]}_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_sha = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", text)
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_b or m_sha.group(1) != kernel_source_sha(kind):
        return None
    return float(m_b.group(1))


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        under_load = [x for x in sm if mx is None or x >= 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(under_load), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- CPU baseline

class OracleSample:
    """The fp64 oracle forward on this host's cores over the last `npos` positions of the
    sequence (all batches and heads) -- a bounded sample of the workload."""

    def __init__(self, w):
        import oracle
        oracle.build()
        self.oracle = oracle
        self.w = w
        self.inp = make_inputs(w, with_dout=False)
        self.cores = oracle.threads()

    def run(self, npos: int) -> float:
        w = self.w
        t0 = time.perf_counter()
        if w.gate:
            gate = gate_weights(w.H, w.d, w.seed + 100)
            self.oracle.fwd_gated(self.inp["q"], self.inp["k"], self.inp["v"], gate, w.k_local,
                                  w.period, w.S, w.mode, rows=(w.N - npos, w.N))
        else:
            self.oracle.fwd(self.inp["q"], self.inp["k"], self.inp["v"], self.inp["alpha"], w.k_local,
                            w.period, w.S, w.mode, rows=(w.N - npos, w.N))
        return time.perf_counter() - t0

    def size_for(self, target_s: float) -> int:
        cal = min(self.w.N, 64)
        t_cal = self.run(cal)
        return int(min(self.w.N, max(cal, cal * target_s / max(t_cal, 1e-6))))

    def describe(self, npos: int) -> str:
        w = self.w
        text = (f"fp64 oracle forward over the last {npos} of {w.N} positions, all {w.B}x{w.H} "
                f"(batch, head) rows; tokens/s = {w.B}*{npos}/t")
        if w.backward:
            text += " (forward only: the oracle backward has no row-range form)"
        return text


class DecodeOracleSample:
    """The fp64 oracle on this host's cores for the decode step of `nb` sequences: row N-1 of
    the forward.  Only the last max(k, S*period) + 1 cache rows can be neighbours of row N-1,
    so the oracle gets that window (the query at its last row), which leaves every key
    distance unchanged."""

    def __init__(self, w):
        import oracle
        oracle.build()
        self.oracle = oracle
        self.w = w
        self.inp = make_inputs(w, with_dout=False)
        self.cores = oracle.threads()
        self.W = min(w.N, max(w.k_local, w.S * w.period) + 1)

    def run(self, nb: int) -> float:
        w, W = self.w, self.W
        q = torch.zeros(nb, w.H, W, w.d, dtype=self.inp["q"].dtype)
        q[:, :, W - 1] = self.inp["q"][:nb]
        a = None
        if self.inp["alpha"] is not None:
            a = torch.full((nb, w.H, W), 0.5, dtype=torch.float32)
            a[:, :, W - 1] = self.inp["alpha"][:nb]
        k = self.inp["k"][:nb, :, w.N - W:].contiguous()
        v = self.inp["v"][:nb, :, w.N - W:].contiguous()
        t0 = time.perf_counter()
        self.oracle.fwd(q, k, v, a, w.k_local, w.period, w.S, w.mode, rows=(W - 1, W))
        return time.perf_counter() - t0

    def size_for(self, target_s: float) -> int:
        t_cal = self.run(1)
        return int(min(self.w.B, max(1, target_s / max(t_cal, 1e-6))))

    def describe(self, nb: int) -> str:
        return (f"fp64 oracle decode step (row N-1 over the last {self.W} cache rows) of {nb} of "
                f"{self.w.B} sequences, all {self.w.H} heads; tokens/s = {nb}/t")


def oracle_sample(w):
    return DecodeOracleSample(w) if w.decode else OracleSample(w)


def tokens_per_unit(w) -> int:
    """Tokens one sample unit stands for: a position of every batch entry, or one sequence."""
    return 1 if w.decode else w.B


def cpu_baseline(w, target_s=10.0):
    """Returns (tokens/s, cores, sample description) of the oracle on a bounded sample."""
    smp = oracle_sample(w)
    n = smp.size_for(target_s)
    t = smp.run(n)
    return tokens_per_unit(w) * n / t, smp.cores, smp.describe(n)


def reduce_max(x: float, world: int, device="cpu") -> float:
    """Max of a per-rank float over all ranks (the slowest rank times the job)."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def reference_arm(args, w, rank, world):
    """The oracle as the reference implementation: rank 0 only, on host cores."""
    if rank != 0:
        return
    smp = oracle_sample(w)
    npos = smp.size_for(min(8.0, 150.0 / (args.warmup + args.steps)))
    for _ in range(args.warmup):
        smp.run(npos)
    per_step = [smp.run(npos) for _ in range(args.steps)]
    value = tokens_per_unit(w) * npos * len(per_step) / sum(per_step)
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * sum(per_step) / len(per_step), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_block(w, "host cores, no GPU"),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": smp.cores,
                             "kind": "oracle", "sample": smp.describe(npos)},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm

def config_block(w, l2_note):
    return {"workload": f"{w.name}: {w.description}", "B": w.B, "H": w.H, "Hkv": w.Hkv, "N": w.N,
            "d": w.d, "k_local": w.k_local, "period": w.period, "S": w.S,
            "mode": {MODE_ECP: "ecp", MODE_PI_BIDIR: "pi_bidir"}.get(w.mode, "pi"),
            "input_dtype": w.dtype, "l2": l2_note}


def roofline_of(w, wk, per_phase):
    """Roofline of the step's dominant kernel: its algorithmic bytes (or useful FLOPs) per launch
    over its mean launch time, against the measured peak that bounds it."""
    peaks, peak_kind = load_peaks()
    dom = max(per_phase, key=lambda n: sum(per_phase[n]))
    dom_ms = statistics.mean(per_phase[dom])
    dom_bytes = wk["bwd_bytes"] if dom == "pi_attn_bwd" else wk["fwd_bytes"]
    dom_flops = wk["bwd_flops"] if dom == "pi_attn_bwd" else wk["fwd_flops"]
    hbm = peaks["hbm_gbs"]
    tensor = peaks["bf16_tflops"]
    t_hbm = dom_bytes / (hbm * 1e9)
    t_tensor = dom_flops / (tensor * 1e12)
    bound = "hbm" if t_hbm >= t_tensor else "tensor"
    if bound == "hbm":
        achieved, peak, unit = dom_bytes / (dom_ms / 1e3) / 1e9, hbm, "GB/s"
    else:
        achieved, peak, unit = dom_flops / (dom_ms / 1e3) / 1e12, tensor, "TFLOP/s"
    traffic = profiled_traffic(w.name, {"pi_attn_fwd": "fwd", "pi_attn_bwd": "bwd",
                                        "pi_attn_decode": "dec"}[dom])
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": traffic, "kernel": dom,
            "peak_source": f"{peak_kind} ({'hbm_gbs' if bound == 'hbm' else 'bf16_tflops'}, burst)",
            "t_roof_us": 1e6 * max(t_hbm, t_tensor), "t_hbm_us": 1e6 * t_hbm,
            "t_tensor_us": 1e6 * t_tensor, "kernel_us": 1e3 * dom_ms,
            "algorithmic_bytes": dom_bytes, "useful_flops": dom_flops,
            "tensor_frac_of_peak": dom_flops / (dom_ms / 1e3) / 1e12 / tensor}


def setup_workload(w, pa, dev, stream):
    """Device inputs and outputs of a workload and the launchers of its step: returns (inputs on
    the host, device tensors, out, lse, gradient buffers, phases), each phase (name, launcher,
    kernels it launches)."""
    inp = make_inputs(w, with_dout=w.backward)
    d = {n: (t.to(dev) if t is not None else None) for n, t in inp.items()}
    return (inp,) + device_set(w, pa, dev, d, stream)


def device_set(w, pa, dev, d, stream):
    """Outputs, gradient buffers and the step's launchers for the device inputs d on `stream`:
    returns (d, out, lse, gradient buffers, phases)."""
    out = torch.empty_like(d["q"])
    lse = torch.empty((w.B, w.H) if w.decode else (w.B, w.H, w.N), device=dev, dtype=torch.float32)
    bufs = {}
    if w.backward:
        bufs = dict(dq=torch.empty_like(d["q"]), dk=torch.empty_like(d["k"]),
                    dv=torch.empty_like(d["v"]),
                    dalpha=torch.empty((w.B, w.H, w.N), device=dev, dtype=torch.float32),
                    ws=torch.empty(max(16, pa.bwd_workspace_size(w.B, w.H, w.Hkv, w.N, w.d)),
                                   device=dev, dtype=torch.uint8))
    gate = alpha_buf = None
    if w.gate:  # the gate's weights are parameters, resident like the model's
        gate = tuple(t.to(dev) for t in gate_weights(w.H, w.d, w.seed + 100))
        alpha_buf = torch.empty((w.B, w.H, w.N), device=dev, dtype=torch.float32)

    def fwd():
        if w.gate:
            pa.fwd_gated(d["q"], d["k"], d["v"], gate, w.k_local, w.period, w.S, w.mode, out=out,
                         lse=lse, alpha_out=alpha_buf, stream=stream)
        else:
            pa.fwd(d["q"], d["k"], d["v"], d["alpha"], w.k_local, w.period, w.S, w.mode, out=out,
                   lse=lse, stream=stream)

    def bwd():
        pa.bwd(d["q"], d["k"], d["v"], d["alpha"], out, lse, d["dout"], w.k_local, w.period, w.S,
               w.mode, dq=bufs["dq"], dk=bufs["dk"], dv=bufs["dv"], dalpha=bufs["dalpha"],
               workspace=bufs["ws"], stream=stream)

    def dec():
        pa.decode(d["q"], d["k"], d["v"], d["alpha"], w.k_local, w.period, w.S, w.mode, out=out,
                  lse=lse, stream=stream)

    if w.decode:
        phases = [("pi_attn_decode", dec, 1)]
    else:
        # the backward is two kernels (query-major dq pass, key-major dk/dv pass) on either path
        phases = [("pi_attn_fwd", fwd, 1)] + ([("pi_attn_bwd", bwd, 2)] if w.backward else [])
    return d, out, lse, bufs, phases


def time_steps(w, pa, dev, stream, phases, steps, warmup, sampler=None, world=1):
    """CUDA-event times (ms) per phase of `steps` steps after `warmup` untimed ones, with the L2
    flushed between steps (outside the events) when a step moves less than twice the L2.  The
    timed steps are bracketed by a barrier (under torchrun) and a device synchronisation; the
    clock sampler, if any, runs over them."""
    wk = work(w, w.backward)
    flush = wk["bytes"] < 2 * L2_BYTES
    scratch = torch.empty(2 * L2_BYTES // 4, device=dev, dtype=torch.float32) if flush else None

    def settle():
        # The flush, then a device-side spin of about 50 us: the host queues the step's events and
        # launches while the device is still busy, so that the events time the kernels and not
        # the host's launch latency between the start event and the first kernel.
        scratch.zero_()
        torch.cuda._sleep(SPIN_CYCLES)

    def step(record=None):
        for name, fn, _ in phases:
            if record is not None:
                record[name][0].record(stream)
            fn()
            if record is not None:
                record[name][1].record(stream)

    for _ in range(warmup):
        if flush:
            settle()
        step()
    torch.cuda.synchronize(dev)
    if pa.status() != 0:
        raise RuntimeError(f"{w.name}: device status word set during warm-up")
    if sampler:
        sampler.start()
    ev = [{n: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for n, _, _ in phases} for _ in range(steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    for k in range(steps):
        if flush:
            settle()
        step(ev[k])
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    status = pa.status()
    if status != 0:
        raise RuntimeError(f"{w.name}: device status word {status} after the timed region")
    return {n: [e[n][0].elapsed_time(e[n][1]) for e in ev] for n, _, _ in phases}


def time_l2_warm(pa, dev, stream, phases, steps=50, warmup=3):
    """Mean ms per step of `steps` steps run back to back with no flush between them (the L2-warm
    figure of a workload small enough to stay in L2), from one event pair around them all."""
    def step():
        for _, fn, _ in phases:
            fn()
    for _ in range(warmup):
        step()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if pa.status() != 0:
        raise RuntimeError("device status word set during the L2-warm steps")
    return e0.elapsed_time(e1) / steps


def step_times(per_phase, steps):
    """Per-step times (ms): the sum over the phases of each step."""
    return [sum(v[k] for v in per_phase.values()) for k in range(steps)]


def config_numbers(w, per_phase, steps, l2_warm_ms=None):
    """The metric's numbers for one workload from its per-phase times."""
    wk = work(w, w.backward)
    total_ms = sum(sum(v) for v in per_phase.values())
    tokens = w.B if w.decode else w.B * w.N
    roof = roofline_of(w, wk, per_phase)
    extra = {"l2_warm_ms_per_step": l2_warm_ms} if l2_warm_ms is not None else {}
    return {"workload": f"{w.name}: {w.description}", "dtype": w.dtype,
            "ms_per_step": total_ms / steps, **extra,
            "median_ms_per_step": statistics.median(step_times(per_phase, steps)),
            "tokens_per_s": tokens * steps / (total_ms / 1e3),
            "useful_tflops": wk["flops"] * steps / (total_ms / 1e3) / 1e12,
            "per_phase_ms": {n: statistics.mean(v) for n, v in per_phase.items()},
            "roofline": {k: roof[k] for k in ("bound", "kernel", "achieved", "peak", "unit", "frac",
                                               "t_roof_us", "kernel_us", "peak_source")},
            "steps": steps}


def other_configs(args, pa, dev, stream, names):
    """The metric's other configurations, each timed in this process after the headline; a step
    is the forward (C5: forward and backward), as for the headline."""
    res = {}
    for name in names:
        w = WORKLOADS[name]
        phases = setup_workload(w, pa, dev, stream)[5]
        per_phase = time_steps(w, pa, dev, stream, phases, args.per_config_steps, 5)
        warm = (time_l2_warm(pa, dev, stream, phases, args.per_config_steps)
                if work(w, w.backward)["bytes"] < 2 * L2_BYTES else None)
        res[name] = config_numbers(w, per_phase, args.per_config_steps, warm)
        del phases
        torch.cuda.empty_cache()
    return res


def gpu_arm(args, w, rank, world, local_rank):
    import structured_sparse_long_gb300 as pa
    from structured_sparse_long_gb300 import build as pbuild

    if rank == 0 or not os.path.exists(pbuild.LIB_PATH):
        pbuild.build()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pa.load()
    stream = torch.cuda.current_stream(dev)

    inp, d, out, lse, bufs, phases = setup_workload(w, pa, dev, stream)
    wk = work(w, w.backward)
    flush = wk["bytes"] < 2 * L2_BYTES
    l2_note = ("L2 flushed between steps (write of a 2x L2 buffer, then a 50 us device-side spin, "
               "outside the timed events)"
               if flush else f"inputs larger than L2 ({wk['bytes'] / 1e6:.0f} MB moved per step)")

    def step():
        for _, fn, _ in phases:
            fn()

    sampler = ClockSampler(local_rank) if rank == 0 else None
    per_phase = time_steps(w, pa, dev, stream, phases, args.steps, args.warmup, sampler=sampler,
                           world=world)
    clocks = sampler.stop() if sampler else None
    l2_warm = (time_l2_warm(pa, dev, stream, phases, min(args.steps, 200))
               if rank == 0 and wk["bytes"] < 2 * L2_BYTES else None)
    step_ms = [sum(per_phase[n][k] for n, _, _ in phases) for k in range(args.steps)]
    total_ms = sum(step_ms)
    total_ms = reduce_max(total_ms, world, dev if args.backend == "nccl" else "cpu")
    ms_per_step = total_ms / args.steps
    tokens_per_step = (w.B if w.decode else w.B * w.N) * world
    value = tokens_per_step * args.steps / (total_ms / 1e3)
    tflops = wk["flops"] * world * args.steps / (total_ms / 1e3) / 1e12

    # dominant kernel roofline (forward kernel: the whole step for the forward workloads)
    roofline = roofline_of(w, wk, per_phase)

    # End to end through the public API with pinned host buffers, as a stream of steps: every
    # step copies its inputs to the device, runs, and copies its outputs back; two device buffer
    # sets let step s+1's inputs travel (host to device) while step s runs and its outputs travel
    # back (device to host), on three streams ordered by events.  (One copy stream per direction
    # measured fastest: splitting the copies over 2, 4 or 8 streams ran 3-9 % slower at C4.)
    e2e = None
    if not args.no_e2e:
        if w.decode:  # per step: the new queries and gates, and the new token's K/V rows
            host = {"q": inp["q"], "alpha": inp["alpha"],
                    "k_new": inp["k"][:, :, w.N - 1].contiguous(),
                    "v_new": inp["v"][:, :, w.N - 1].contiguous()}
            host = {n: (t.pin_memory() if t is not None else None) for n, t in host.items()}
        else:
            host = {n: (t.pin_memory() if t is not None else None) for n, t in inp.items()}
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for n, t in host.items()
                  if t is not None and (n != "dout" or w.backward))
        d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()
        grads_h = {}
        if w.backward:
            grads_h = {n: torch.empty(bufs[n].shape, dtype=bufs[n].dtype).pin_memory()
                       for n in ("dq", "dk", "dv", "dalpha")}
            d2h += sum(t.numel() * t.element_size() for t in grads_h.values())
        s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        d2 = {n: (t.clone() if t is not None else None) for n, t in d.items()}
        sets = [(d, out, lse, bufs, phases), device_set(w, pa, dev, d2, stream)]
        torch.cuda.synchronize(dev)
        ev_in = [torch.cuda.Event() for _ in sets]    # the set's inputs landed
        ev_run = [torch.cuda.Event() for _ in sets]   # its step ran (inputs read, outputs written)
        ev_back = [torch.cuda.Event() for _ in sets]  # its outputs copied back

        def e2e_step(k):
            b = k % 2
            dd, o, ls, bf, ph = sets[b]
            if k >= 2:
                s_h2d.wait_event(ev_run[b])
            with torch.cuda.stream(s_h2d):
                for n, t in host.items():
                    if t is None or (n == "dout" and not w.backward):
                        continue
                    if n in ("k_new", "v_new"):  # append the new token to the cache (row N-1)
                        dd[n[0]][:, :, w.N - 1].copy_(t, non_blocking=True)
                    else:
                        dd[n].copy_(t, non_blocking=True)
            ev_in[b].record(s_h2d)
            stream.wait_event(ev_in[b])
            if k >= 2:
                stream.wait_event(ev_back[b])
            for _, fn, _ in ph:
                fn()
            ev_run[b].record(stream)
            s_d2h.wait_event(ev_run[b])
            with torch.cuda.stream(s_d2h):
                out_h.copy_(o, non_blocking=True)
                lse_h.copy_(ls, non_blocking=True)
                for n, t in grads_h.items():
                    t.copy_(bf[n], non_blocking=True)
            ev_back[b].record(s_d2h)

        for k in range(max(2, min(args.warmup, 3))):
            e2e_step(k)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_e2e = max(2, min(args.steps, 10))
        e0.record(s_h2d)
        for k in range(n_e2e):
            e2e_step(k)
        e1.record(s_d2h)  # after the last step's copy back (the stream is in order)
        torch.cuda.synchronize(dev)
        e_ms = e0.elapsed_time(e1)
        e_ms = reduce_max(e_ms, world, dev if args.backend == "nccl" else "cpu")
        e2e = {"value": tokens_per_step * n_e2e / (e_ms / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e_ms / n_e2e, "steps": n_e2e,
               "pipelining": "two device buffer sets; host-to-device copies, the step and the "
                             "device-to-host copies on three streams, so step s+1's inputs travel "
                             "while step s runs"}
        del sets, d2
        torch.cuda.empty_cache()

    if rank != 0:
        return
    per_config = None
    if w.name == "C4" and not args.no_per_config:  # the metric's other configurations
        per_config = {"C4": config_numbers(w, per_phase, args.steps)}
        per_config.update(other_configs(args, pa, dev, stream, ("C1", "C2", "C3", "C5")))
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        tps, cores, desc = cpu_baseline(w, target_s=args.cpu_seconds)
        cpu = {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc}
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "median_ms_per_step": statistics.median(step_ms),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic (seeded torch.Generator, shapes of the workload)",
            "config": config_block(w, l2_note), "useful_tflops": tflops,
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": args.steps * sum(n for _, _, n in phases),
            "clocks": clocks, "per_phase_ms": {n: statistics.mean(v) for n, v in per_phase.items()},
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}
    if l2_warm is not None:  # the same steps back to back, L2 not flushed (rank 0's own)
        line["l2_warm_ms_per_step"] = l2_warm
    if per_config is not None:
        line["per_config"] = per_config
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="C4", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--backend", default="nccl", choices=["nccl", "gloo"])
    ap.add_argument("--no-per-config", action="store_true",
                    help="the default C4 run also times C1, C2, C3 and C5; this skips them")
    ap.add_argument("--per-config-steps", type=int, default=30)
    ap.add_argument("--seq", type=int, default=0,
                    help="override the sequence length N (smaller cases for profiler captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = WORKLOADS[args.config]
    if args.seq:
        w = w.replace(N=args.seq, name=f"{w.name}-N{args.seq}",
                      description=w.description + f" (N overridden to {args.seq})")
    if args.impl == "reference":
        reference_arm(args, w, rank, world)
        return
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group(args.backend)
    try:
        gpu_arm(args, w, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
