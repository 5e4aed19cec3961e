#!/usr/bin/env python
"""Benchmark of the M2RNN forward + backward-through-time scans on GB300.

One step = one pass of the whole hot path over one batch of seeded synthetic
input: the forward scan (writing the per-chunk checkpoints) followed by the
backward scan that reuses them, for the bf16 forward+backward workload
B=4, heads=8, T=4096, K=V=64.  ``value`` is tokens*heads/s (B*T*heads per
step / device time) with inputs resident in HBM; ``e2e`` is the same through
the C ABI with host buffers (pinned host->device copies of the inputs and
device->host copies of every result inside the timed region).  The forward-
only workloads (T=2048 K=V=64, T=4096 K=V=128, T=16384 K=V=64) are timed too
and reported under ``forward``.

``--impl reference`` times the float64 CPU oracle on the same workload
(a bounded sample per step) instead.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
Under torchrun every rank runs its own full batch (independent chains, no
data-path collective: weak scaling); timing is the max over ranks.
"""
from __future__ import annotations

import os

_CORES = os.cpu_count() or 1
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(_CORES))
os.environ.setdefault("OMP_NUM_THREADS", str(_CORES))

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import threading  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from matrix_state_non_gb300.inputs import (WORKLOADS, make_gate_inputs, make_norm_inputs,  # noqa: E402
                                           make_workload)

METRIC = "M²RNN scan tokens·heads/s (fwd, fwd+bwd) and % of tensor/HBM roofline, 1 GB300"
UNIT = "tokens*heads/s"
MAIN = "fwdbwd_bf16_k64"
FWD_EXTRA = ("fwd_bf16_k64", "fwd_bf16_k128", "fwd_bf16_16k", "mv_bf16_k64v16")
IN_NAMES = ("q", "k", "v", "f", "W", "w_r")
GRADS = ("dq", "dk", "dv", "df", "dW", "dw_r")
CKPT_EVERY = 20  # chunk length of the V = 64 backward rebuild (its longest: shared-memory bound)
CKPT_EVERY_MV = 20  # the V = 16 pipelined backward's longest chunk (its TMEM chunk cache is double-buffered)
CKPT_EVERY_K128 = 8  # the K = V = 128 backward: its chunk cache (64 KB per step and chain) stays in L2
FLUSH_BYTES = 256 << 20  # larger than the 129 MB L2


# ---------------------------------------------------------------------------
# Shared helpers
# ---------------------------------------------------------------------------
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm_gbs=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


def units(w):
    return w["B"] * w["T"] * w["N"]


def fwd_flops(w):
    return 2.0 * w["K"] * w["V"] ** 2 * units(w)


def bwd_flops(w):
    return 4.0 * w["K"] * w["V"] ** 2 * units(w)


def qk_share(w):
    """Fraction of the q/k traffic per unit: 1/N when one q/k serves every head."""
    return 1.0 / w["N"] if w.get("shared_qk") else 1.0


def io_bytes_fwd(w, s_in=2):
    K, V = w["K"], w["V"]
    return units(w) * ((2 * K * qk_share(w) + V + 1) * s_in + 4 * V)


def io_bytes_bwd(w, s_in=2, ckpt_every=CKPT_EVERY):
    K, V = w["K"], w["V"]
    per_unit = (2 * K * qk_share(w) + V + 1) * s_in + 4 * V + 4 * (2 * K * qk_share(w) + V + 1)
    ck = 4.0 * K * V * units(w) / ckpt_every
    return units(w) * per_unit + ck


def stash_bytes(w):
    """The forward's fp16 Z stash (written by the forward, read by the
    backward of a training step): 2 K V bytes per unit."""
    return 2.0 * w["K"] * w["V"] * units(w)


# The sources each profiled kernel is built from: a recorded DRAM traffic
# figure is used only while these files are unchanged.
KERNEL_SOURCES = {
    "m2rnn_backward": ("mma_backward.cu", "mma_common.cuh", "ptx.cuh", "gate.cuh", "internal.h", "status.cuh"),
    "m2rnn_forward": ("mma_forward.cu", "tc_forward.cu", "mv_forward.cu", "mma_common.cuh", "ptx.cuh",
                      "gate.cuh", "internal.h", "status.cuh"),
}


def source_hash(kernel: str = None):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "matrix_state_non_gb300", "csrc")
    names = KERNEL_SOURCES.get(kernel) or sorted(os.listdir(csrc))
    for name in sorted(names):
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(name.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh)
    except (OSError, ValueError):
        return None
    ent = rec.get(f"{kernel}@{workload}")
    if not ent or ent.get("source_hash") != source_hash(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
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
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# Distributed plumbing (torchrun): barrier + max over ranks
# ---------------------------------------------------------------------------
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as td
            backend = "nccl" if _cuda_ok() else "gloo"
            td.init_process_group(backend=backend)
            self.pg = td

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        dev = "cuda" if _cuda_ok() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def _cuda_ok():
    import torch
    return torch.cuda.is_available()


# ---------------------------------------------------------------------------
# Reference arm: the float64 CPU oracle on a bounded sample of the workload
# ---------------------------------------------------------------------------
def run_reference(args, dist):
    if dist.rank != 0:
        return None
    from oracle import backward as oracle_backward
    from oracle import forward as oracle_forward
    w = WORKLOADS[MAIN]
    t_sample = 256  # timesteps of every chain per step: a few seconds of CPU work
    inp = make_workload(MAIN)
    ex = inp.exact
    sl = slice(0, t_sample)
    a = [ex["q"][:, sl], ex["k"][:, sl], ex["v"][:, sl], ex["f"][:, sl], ex["W"], ex["w_r"]]
    dy = ex["dy"][:, sl]

    def step():
        oracle_forward(*a)
        oracle_backward(*a, dy)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    n_units = w["B"] * w["N"] * t_sample
    val = n_units / dt
    cores = int(os.environ.get("OPENBLAS_NUM_THREADS", _CORES))
    sample = (f"all {w['B']}x{w['N']} chains, first {t_sample} of {w['T']} steps, "
              "forward + backward (float64 numpy oracle)")
    return {
        "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOADS[MAIN]["desc"], "B": w["B"], "T": w["T"], "heads": w["N"],
                   "K": w["K"], "V": w["V"], "parallelism": "cpu"},
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def cpu_baseline_sample():
    """The oracle as it stands on a bounded sample of the main workload."""
    from oracle import backward as oracle_backward
    from oracle import forward as oracle_forward
    w = WORKLOADS[MAIN]
    t_sample = 512
    inp = make_workload(MAIN)
    ex = inp.exact
    sl = slice(0, t_sample)
    a = [ex["q"][:, sl], ex["k"][:, sl], ex["v"][:, sl], ex["f"][:, sl], ex["W"], ex["w_r"]]
    t0 = time.perf_counter()
    oracle_forward(*a)
    oracle_backward(*a, ex["dy"][:, sl])
    dt = time.perf_counter() - t0
    n_units = w["B"] * w["N"] * t_sample
    return {"value": n_units / dt, "unit": UNIT,
            "cores": int(os.environ.get("OPENBLAS_NUM_THREADS", _CORES)), "kind": "oracle",
            "sample": (f"all {w['B']}x{w['N']} chains, first {t_sample} of {w['T']} steps, "
                       f"forward + backward, {dt:.1f} s of float64 numpy")}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_gpu(args, dist):
    import torch

    from matrix_state_non_gb300 import binding

    torch.cuda.set_device(dist.local)
    dev = torch.device("cuda", dist.local)
    binding.load()
    pk = peaks()
    w = WORKLOADS[MAIN]
    inp = make_workload(MAIN)
    d = binding.to_device(inp, dev)
    B, T, N, K, V = w["B"], w["T"], w["N"], w["K"], w["V"]
    stream = torch.cuda.current_stream(dev)
    # Preallocated outputs and workspaces.  The forward leaves its Z stash
    # (fp16 Z_t of every step) and checkpoints for the backward.
    fwd_out = binding.forward(*(d[n] for n in IN_NAMES), ckpt_every=CKPT_EVERY, stash=True)
    bwd_out = binding.backward(*(d[n] for n in IN_NAMES), d["dy"], ckpt=fwd_out["ckpt"],
                               ckpt_every=CKPT_EVERY, z_stash=fwd_out["z_stash"])
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def step(timing=None):
        if timing is not None:
            timing[0].record(stream)
        binding.forward(*(d[n] for n in IN_NAMES), ckpt_every=CKPT_EVERY, stash=True, out=fwd_out,
                        workspace=fwd_out["workspace"])
        if timing is not None:
            timing[1].record(stream)
        binding.backward(*(d[n] for n in IN_NAMES), d["dy"], ckpt=fwd_out["ckpt"],
                         ckpt_every=CKPT_EVERY, z_stash=fwd_out["z_stash"], out=bwd_out,
                         workspace=bwd_out["workspace"])
        if timing is not None:
            timing[2].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    st, detail = binding.sync_status(bwd_out["workspace"])
    if st != binding.M2RNN_OK:
        raise RuntimeError(f"device status {binding.status_string(st)} at {detail}")

    sampler = ClockSampler(torch.cuda.current_device()) if dist.rank == 0 else None
    timings = [(ev(), ev(), ev()) for _ in range(args.steps)]
    dist.barrier()
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.start()
        time.sleep(0.3)
    for i in range(args.steps):
        flush.zero_()  # L2 flush between timed steps (outside the events)
        step(timings[i])
    torch.cuda.synchronize(dev)
    clocks = sampler.stop() if sampler else None
    dist.barrier()
    fwd_ms = [a.elapsed_time(b) for a, b, _ in timings]
    bwd_ms = [b.elapsed_time(c) for _, b, c in timings]
    step_ms_local = sum(f + b for f, b in zip(fwd_ms, bwd_ms)) / args.steps
    step_ms = dist.max(step_ms_local)
    value = dist.world * units(w) / (step_ms * 1e-3)

    # e2e: host buffers through the C ABI, every step's copies inside the
    # timed region: H2D of the step's inputs from pinned memory, the step,
    # D2H of its outputs (y and every gradient).  Steps are pipelined as a
    # training loop would run them: two device buffer sets, the H2D of step
    # i + 1 and the D2H of step i - 1 on their own streams while step i
    # computes.  The per-step working set (the 1 GB Z stash) exceeds L2, so
    # no flush is interposed.
    names_in = list(IN_NAMES) + ["dy"]
    host_in = {n: torch.empty_like(d[n], device="cpu").pin_memory() for n in names_in}
    for n in host_in:
        host_in[n].copy_(d[n].cpu())
    sets = []
    for _ in range(2):
        dd = {n: torch.empty_like(d[n]) for n in names_in}
        fo = binding.forward(*(d[n] for n in IN_NAMES), ckpt_every=CKPT_EVERY, stash=True)
        bo = binding.backward(*(d[n] for n in IN_NAMES), d["dy"], ckpt=fo["ckpt"], ckpt_every=CKPT_EVERY,
                              z_stash=fo["z_stash"])
        sets.append((dd, fo, bo))
    n_out = 1 + len(GRADS)
    host_out = [[torch.empty_like(t, device="cpu").pin_memory() for t in [fo["y"]] + [bo[g] for g in GRADS]]
                for _, fo, bo in sets]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [ev(), ev()]
    ev_done = [ev(), ev()]
    ev_out = [ev(), ev()]
    for e_ in ev_done + ev_out:
        e_.record(stream)

    def e2e_run(nsteps):
        for i in range(nsteps):
            k_ = i % 2
            dd, fo, bo = sets[k_]
            with torch.cuda.stream(s_h2d):
                s_h2d.wait_event(ev_done[k_])  # step i - 2 is done with this input set
                for n in names_in:
                    dd[n].copy_(host_in[n], non_blocking=True)
                ev_in[k_].record(s_h2d)
            stream.wait_event(ev_in[k_])
            stream.wait_event(ev_out[k_])  # the D2H of step i - 2 has read this output set
            binding.forward(*(dd[n] for n in IN_NAMES), ckpt_every=CKPT_EVERY, stash=True, out=fo,
                            workspace=fo["workspace"])
            binding.backward(*(dd[n] for n in IN_NAMES), dd["dy"], ckpt=fo["ckpt"], ckpt_every=CKPT_EVERY,
                             z_stash=fo["z_stash"], out=bo, workspace=bo["workspace"])
            ev_done[k_].record(stream)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(ev_done[k_])
                for hd, dv_ in zip(host_out[k_], [fo["y"]] + [bo[g] for g in GRADS]):
                    hd.copy_(dv_, non_blocking=True)
                ev_out[k_].record(s_d2h)

    e2e_run(max(3, args.warmup))
    torch.cuda.synchronize(dev)
    dist.barrier()
    a, b = ev(), ev()
    a.record(s_h2d)
    e2e_run(args.steps)
    with torch.cuda.stream(s_d2h):
        b.record(s_d2h)
    torch.cuda.synchronize(dev)
    for _, fo, bo in sets:
        st, detail = binding.sync_status(bo["workspace"])
        if st != binding.M2RNN_OK:
            raise RuntimeError(f"e2e: device status {binding.status_string(st)} at {detail}")
    assert n_out == len(host_out[0])
    e2e_local = a.elapsed_time(b) / args.steps
    e2e_ms = dist.max(e2e_local)
    e2e_val = dist.world * units(w) / (e2e_ms * 1e-3)

    # Roofline of the dominant kernel in the step, against the burst bf16
    # peak: the kernels run for milliseconds at a small fraction of the
    # tensor pipe, far from the power cap the sustained figure reflects.
    f_avg = sum(fwd_ms) / len(fwd_ms)
    b_avg = sum(bwd_ms) / len(bwd_ms)
    peak = pk["bf16"]
    if b_avg >= f_avg:
        kname, kflops, kms = "m2rnn_backward", bwd_flops(w), b_avg
    else:
        kname, kflops, kms = "m2rnn_forward", fwd_flops(w), f_avg
    achieved = kflops / (kms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": profiled_traffic(kname, MAIN),
                "kernel": kname, "peak_source": f"{pk['source']} bf16 burst",
                "kernel_ms": kms, "ns_per_step_per_chain": kms * 1e6 / T,
                "flop_per_launch": kflops,
                "step_frac": (fwd_flops(w) + bwd_flops(w)) / (step_ms * 1e-3) / 1e12 / peak,
                "hbm_frac": ((io_bytes_bwd(w) if kname == "m2rnn_backward" else io_bytes_fwd(w)) + stash_bytes(w))
                / (kms * 1e-3) / (pk["hbm_gbs"] * 1e9)}

    # Forward-only workloads.
    fwd_extra = {}
    if not args.no_extra:
        for name in FWD_EXTRA:
            fwd_extra[name] = time_forward(name, binding, dev, stream, flush, pk, dist,
                                           reps=max(3, args.steps // 2))
        # The same long-context workload on the tcgen05 kernel, for
        # comparison with the warp-MMA kernel the dispatcher picks.
        with binding.kernel_family("tcgen05"):
            fwd_extra["fwd_bf16_16k@tcgen05"] = time_forward("fwd_bf16_16k", binding, dev, stream, flush,
                                                             pk, dist, reps=3)
        with binding.kernel_family("simt"):  # the multi-value workload on the fp32 kernel, for comparison
            fwd_extra["mv_bf16_k64v16@simt"] = time_forward("mv_bf16_k64v16", binding, dev, stream, flush,
                                                            pk, dist, reps=3)
        fwd_extra["decode_bf16_k64"] = time_decode(binding, dev, stream, dist)
        fwd_extra["mv_bf16_k64v16@fwd+bwd"] = time_fwdbwd("mv_bf16_k64v16", binding, dev, stream, flush, pk,
                                                          dist)
        fwd_extra["gated_block_bf16_k64"] = time_gated_block(binding, dev, stream, flush, pk, dist)
        fwd_extra["fwdbwd_bf16_k128"] = time_fwdbwd("fwdbwd_bf16_k128", binding, dev, stream, flush, pk, dist)
    cpu = cpu_baseline_sample() if (dist.rank == 0 and not args.no_cpu) else None
    launches_per_step = 4  # forward scan, backward scan, dv/df row sums, dW/dw_r partial sums
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w["desc"], "B": B, "T": T, "heads": N, "K": K, "V": V,
                   "state": "fp32", "ckpt_every": CKPT_EVERY,
                   "z_stash": "fp16 Z_t of every step, written by the forward, read by the backward",
                   "l2": "flushed between timed steps (256 MiB write outside the events)",
                   "parallelism": f"replicas x{dist.world} (independent chains, no collective)"},
        "configs": summary_block(w, step_ms, fwd_extra, pk),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "pipelining": "two buffer sets; H2D of step i+1 and D2H of step i-1 on copy streams "
                              "overlap step i; working set larger than L2, no flush"},
        "clocks": clocks,
        "gpu_launches": launches_per_step * args.steps,
        "step_breakdown_ms": {"forward": f_avg, "backward": b_avg},
        "forward": fwd_extra,
        "kernels": {"forward": "warp-mma with readout warps (writes the Z stash)",
                    "backward": "warp-mma chain + tcgen05 dW"},
    }
    return line


def summary_block(w, step_ms, fwd_extra, pk):
    """Compact per-workload figures (ms, ns per step and chain, roofline
    fraction against the burst bf16 peak / HBM copy rate), first in the line."""
    out = {}
    for name in ("fwd_bf16_k64", "fwd_bf16_k128", "fwd_bf16_16k", "fwd_bf16_16k@tcgen05"):
        r = fwd_extra.get(name)
        if r:
            out[name] = {"kernel": r["kernel"], "ms": round(r["ms"], 4),
                         "ns_per_step_per_chain": round(r["ns_per_step_per_chain"], 1),
                         "roofline_frac": round(r["roofline_frac"], 4)}
    fl = fwd_flops(w) + bwd_flops(w)
    out[MAIN] = {"kernel": "warp-mma fwd + warp-mma/tcgen05 bwd", "ms": round(step_ms, 4),
                 "ns_per_step_per_chain": round(step_ms * 1e6 / w["T"], 1),
                 "roofline_frac": round(fl / (pk["bf16"] * 1e12) / (step_ms * 1e-3), 4)}
    return out


def time_forward(name, binding, dev, stream, flush, pk, dist, reps=5):
    import torch
    w = WORKLOADS[name]
    inp = make_workload(name)
    d = binding.to_device(inp, dev)
    out = binding.forward(*(d[n] for n in IN_NAMES))
    for _ in range(3):
        binding.forward(*(d[n] for n in IN_NAMES), out=out, workspace=out["workspace"])
    torch.cuda.synchronize(dev)
    ms = []
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        binding.forward(*(d[n] for n in IN_NAMES), out=out, workspace=out["workspace"])
        b.record(stream)
        ms.append((a, b))
    torch.cuda.synchronize(dev)
    st, detail = binding.sync_status(out["workspace"])
    if st != binding.M2RNN_OK:
        raise RuntimeError(f"{name}: device status {binding.status_string(st)} at {detail}")
    t = dist.max(sum(a.elapsed_time(b) for a, b in ms) / reps)
    fl = fwd_flops(w)
    by = io_bytes_fwd(w)
    t_tensor = fl / (pk["bf16"] * 1e12)
    t_hbm = by / (pk["hbm_gbs"] * 1e9)
    del d, out
    kern = {0: "simt", 1: "tcgen05", 2: "warp-mma"}.get(
        binding.m2rnn_path(w["K"], w["V"], binding.M2RNN_BF16), "?")
    return {"workload": w["desc"], "kernel": kern, "ms": t, "value": dist.world * units(w) / (t * 1e-3), "unit": UNIT,
            "ns_per_step_per_chain": t * 1e6 / w["T"],
            "roofline_ms": max(t_tensor, t_hbm) * 1e3,
            "roofline_frac": max(t_tensor, t_hbm) / (t * 1e-3),
            "bound": "tensor" if t_tensor >= t_hbm else "hbm",
            "tensor_tflops": fl / (t * 1e-3) / 1e12,
            "peak_source": f"{pk['source']} bf16 burst / hbm copy"}


def time_fwdbwd(name, binding, dev, stream, flush, pk, dist, reps=3):
    """Forward (writing checkpoints) + backward of a training workload, per
    step: the same protocol as the headline step, for another workload."""
    import torch
    w = WORKLOADS[name]
    C = CKPT_EVERY_MV if w["V"] == 16 else (CKPT_EVERY_K128 if w["V"] == 128 else CKPT_EVERY)
    # The Z stash where the shape has one (V = 64, V = 16).
    stash = binding.m2rnn_z_stash_size(w["B"], w["T"], w["N"], w["K"], w["V"], binding.M2RNN_BF16) > 0
    inp = make_workload(name)
    d = binding.to_device(inp, dev)
    fo = binding.forward(*(d[n] for n in IN_NAMES), ckpt_every=C, stash=stash)
    bo = binding.backward(*(d[n] for n in IN_NAMES), d["dy"], ckpt=fo["ckpt"], ckpt_every=C,
                          z_stash=fo.get("z_stash"))

    def step():
        binding.forward(*(d[n] for n in IN_NAMES), ckpt_every=C, stash=stash, out=fo,
                        workspace=fo["workspace"])
        binding.backward(*(d[n] for n in IN_NAMES), d["dy"], ckpt=fo["ckpt"], ckpt_every=C,
                         z_stash=fo.get("z_stash"), out=bo, workspace=bo["workspace"])

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    ev = []
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        ev.append((a, b))
    torch.cuda.synchronize(dev)
    for out in (fo, bo):
        st, detail = binding.sync_status(out["workspace"])
        if st != binding.M2RNN_OK:
            raise RuntimeError(f"{name}: device status {binding.status_string(st)} at {detail}")
    t = dist.max(sum(a.elapsed_time(b) for a, b in ev) / reps)
    fl = fwd_flops(w) + bwd_flops(w)
    t_tensor = fl / (pk["bf16"] * 1e12)
    t_hbm = (io_bytes_fwd(w) + io_bytes_bwd(w, ckpt_every=C) + (2 * stash_bytes(w) if stash else 0)) / \
        (pk["hbm_gbs"] * 1e9)
    del d, fo, bo
    kern = {16: "warp-mma (V = 16: compute/readout forward, rebuild/chain backward)", 64: "warp-mma forward (readout warps), warp-mma chain + tcgen05 dW backward",
            128: "tcgen05 forward, tcgen05 backward (chain, dW, dk, dv, dq)"}.get(w["V"], "?")
    return {"workload": w["desc"] + (", Z stash" if stash else "") + f", checkpoints every {C}",
            "kernel": kern, "ms": t,
            "value": dist.world * units(w) / (t * 1e-3), "unit": UNIT,
            "ns_per_step_per_chain": t * 1e6 / w["T"],
            "roofline_ms": max(t_tensor, t_hbm) * 1e3, "roofline_frac": max(t_tensor, t_hbm) / (t * 1e-3),
            "bound": "tensor" if t_tensor >= t_hbm else "hbm"}


def time_gated_block(binding, dev, stream, flush, pk, dist, reps=3):
    """The fwd+bwd workload with the forget gate computed in the scan kernels
    from (a, alpha, beta) and the gated RMSNorm output path around it: gated
    forward, output norm, its backward (whose dy feeds the scan), gated
    backward (da, dalpha, dbeta).  Each piece timed with events inside one
    step; the two norm kernels also timed alone after an L2 flush, against
    the HBM roofline of their algorithmic bytes."""
    import torch
    w = WORKLOADS[MAIN]
    B, T, N, K, V = w["B"], w["T"], w["N"], w["K"], w["V"]
    inp = make_workload(MAIN)
    d = binding.to_device(inp, dev)
    gs, _ = make_gate_inputs(B, T, N, "bf16", seed=w["seed"] + 100)
    ns, _ = make_norm_inputs(B, T, N, V, "bf16", seed=w["seed"] + 101)
    up = {n: binding.to_device(_Store(x), dev)["x"] for n, x in list(gs.items()) + list(ns.items())}
    gate = (up["a"], up["alpha"], up["beta"])
    args = (d["q"], d["k"], d["v"], None, d["W"], d["w_r"])
    fo = binding.forward(*args, gate=gate, ckpt_every=CKPT_EVERY, stash=True)
    out = binding.output_norm(fo["y"], up["g"], up["w"])
    nb = binding.output_norm_backward(fo["y"], up["g"], up["w"], up["dout"])
    bo = binding.backward(*args, nb["dy"], gate=gate, ckpt=fo["ckpt"], ckpt_every=CKPT_EVERY,
                          z_stash=fo["z_stash"])
    nws = torch.empty(binding.m2rnn_output_norm_backward_workspace_size(B, T, N, V), device=dev,
                      dtype=torch.uint8)

    def norm_fwd():
        binding.output_norm(fo["y"], up["g"], up["w"], out=out)

    def norm_bwd():
        binding.output_norm_backward(fo["y"], up["g"], up["w"], up["dout"], out=nb, workspace=nws)

    def step(evs=None):
        rec = (lambda i: evs[i].record(stream)) if evs else (lambda i: None)
        rec(0)
        binding.forward(*args, gate=gate, ckpt_every=CKPT_EVERY, stash=True, out=fo, workspace=fo["workspace"])
        rec(1)
        norm_fwd()
        rec(2)
        norm_bwd()
        rec(3)
        binding.backward(*args, nb["dy"], gate=gate, ckpt=fo["ckpt"], ckpt_every=CKPT_EVERY,
                         z_stash=fo["z_stash"], out=bo, workspace=bo["workspace"])
        rec(4)

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    runs = []
    for _ in range(reps):
        flush.zero_()
        evs = [mk() for _ in range(5)]
        step(evs)
        runs.append(evs)
    alone = {}
    # After the write flush, read another buffer larger than L2: that writes
    # the flush's dirty lines back before the timed launch instead of during
    # it (a kernel of ~20 us would otherwise pay for them).
    evict = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    for name, fn in (("norm_fwd", norm_fwd), ("norm_bwd", norm_bwd)):
        pairs = []
        for _ in range(reps):
            flush.zero_()
            evict.sum()
            a, b = mk(), mk()
            a.record(stream)
            fn()
            b.record(stream)
            pairs.append((a, b))
        alone[name] = pairs
    torch.cuda.synchronize(dev)
    for o in (fo, bo):
        st, detail = binding.sync_status(o["workspace"])
        if st != binding.M2RNN_OK:
            raise RuntimeError(f"gated block: device status {binding.status_string(st)} at {detail}")
    piece = lambda i: dist.max(sum(e[i].elapsed_time(e[i + 1]) for e in runs) / reps)  # noqa: E731
    ms = {"gated_forward": piece(0), "norm_forward": piece(1), "norm_backward": piece(2),
          "gated_backward": piece(3)}
    total = sum(ms.values())
    elems = B * T * N * V
    nbytes = {"norm_fwd": elems * (4 + 2 + 4) + N * V * 4, "norm_bwd": elems * (4 + 2 + 4 + 4 + 4) + N * V * 4}
    alone_ms = {k: dist.max(sum(a.elapsed_time(b) for a, b in v) / reps) for k, v in alone.items()}
    norm = {k: {"ms": alone_ms[k], "bytes": nbytes[k],
                "achieved_gbs": nbytes[k] / (alone_ms[k] * 1e-3) / 1e9,
                "hbm_frac": nbytes[k] / (alone_ms[k] * 1e-3) / (pk["hbm_gbs"] * 1e9)} for k in alone_ms}
    del d, fo, bo, out, nb, evict
    return {"workload": w["desc"] + ", gate from (a, alpha, beta) in-kernel, RMSNorm(y*g) over N*V",
            "ms": total, "value": dist.world * units(w) / (total * 1e-3), "unit": UNIT, "pieces_ms": ms,
            "norm_alone_after_l2_flush": norm}


class _Store:
    """Adapter so binding.to_device uploads one array."""

    def __init__(self, x):
        self.store = {"x": x}


def time_decode(binding, dev, stream, dist, steps=64):
    """One-token decoding (m2rnn_decode_step): the B x heads states of the
    forward+backward workload advanced one step per call, `steps` calls in a
    row, the state updated in place.  Timed twice: called eagerly from Python
    (bound by the host call) and replayed as one CUDA graph of the `steps`
    calls (the device time per step)."""
    import torch
    w = WORKLOADS[MAIN]
    inp = make_workload(MAIN)
    d = binding.to_device(inp, dev)
    B, N, K, V = w["B"], w["N"], w["K"], w["V"]
    toks = [[d[n][:, t].contiguous() for n in ("q", "k", "v", "f")] for t in range(steps)]
    H = torch.zeros((B, N, K, V), device=dev, dtype=torch.float32)
    y = torch.empty((B, N, V), device=dev, dtype=torch.float32)
    ws = torch.empty(binding.m2rnn_forward_workspace_size(B, 1, N, K, V, binding.M2RNN_BF16),
                     device=dev, dtype=torch.uint8)

    def run_all():
        for t in range(steps):
            binding.decode_step(H, *toks[t], d["W"], d["w_r"], y=y, workspace=ws)

    for t in range(8):
        binding.decode_step(H, *toks[t], d["W"], d["w_r"], y=y, workspace=ws)
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    run_all()
    b.record(stream)
    torch.cuda.synchronize(dev)
    us_eager = dist.max(a.elapsed_time(b) * 1e3 / steps)
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        run_all()  # warm the side stream before capture
    torch.cuda.current_stream(dev).wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run_all()
    graph.replay()
    torch.cuda.synchronize(dev)
    reps = 5
    a.record(stream)
    for _ in range(reps):
        graph.replay()
    b.record(stream)
    torch.cuda.synchronize(dev)
    us = dist.max(a.elapsed_time(b) * 1e3 / (reps * steps))
    st, detail = binding.sync_status(ws)
    if st != binding.M2RNN_OK:
        raise RuntimeError(f"decode: device status {binding.status_string(st)} at {detail}")
    return {"workload": f"bf16 decode, {B}x{N} states of {K}x{V}, one token per call, {steps} calls",
            "kernel": "decode kernel (warp MMA, state in registers)", "us_per_step": us,
            "us_per_step_eager": us_eager, "timing": "CUDA graph of the calls (eager: Python call per step)",
            "value": dist.world * B * N / (us * 1e-6), "unit": UNIT, "launches_per_step": 1}


def run_only(args, dist):
    """One workload, no extras: warm-up launches, then --steps launches."""
    import torch

    from matrix_state_non_gb300 import binding
    torch.cuda.set_device(dist.local)
    dev = torch.device("cuda", dist.local)
    w = WORKLOADS[args.only]
    inp = make_workload(args.only)
    d = binding.to_device(inp, dev)
    ck = (CKPT_EVERY_MV if w["V"] == 16 else (CKPT_EVERY_K128 if w["V"] == 128 else CKPT_EVERY)) if w["backward"] else 0
    # Training workloads run as the benchmark step does: with the Z stash where the shape has one.
    stash = w["backward"] and binding.m2rnn_z_stash_size(w["B"], w["T"], w["N"], w["K"], w["V"],
                                                         binding.M2RNN_BF16 if w["dtype"] == "bf16"
                                                         else binding.M2RNN_F32) > 0
    out = binding.forward(*(d[n] for n in IN_NAMES), ckpt_every=ck, stash=stash)
    bout = None

    def step():
        nonlocal bout
        binding.forward(*(d[n] for n in IN_NAMES), ckpt_every=ck, stash=stash, out=out,
                        workspace=out["workspace"])
        if w["backward"]:
            bout = binding.backward(*(d[n] for n in IN_NAMES), d["dy"], ckpt=out["ckpt"],
                                    ckpt_every=ck, z_stash=out.get("z_stash"), out=bout,
                                    workspace=None if bout is None else bout["workspace"])

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize(dev)
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    st, detail = binding.sync_status(out["workspace"])
    return {"only": args.only, "host_ms_per_step": dt * 1e3, "status": binding.status_string(st),
            "detail": detail}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    ap.add_argument("--no-extra", action="store_true", help="skip the forward-only workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--only", choices=sorted(WORKLOADS), default=None,
                    help="run just this workload (forward, or forward+backward) --steps times "
                         "after --warmup; for profiler captures")
    args = ap.parse_args()
    dist = Dist()
    try:
        if args.only:
            line = run_only(args, dist)
        elif args.impl == "reference":
            line = run_reference(args, dist)
        else:
            line = run_gpu(args, dist)
        if dist.rank == 0 and line is not None:
            print(json.dumps(line), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
