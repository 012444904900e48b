#!/usr/bin/env python3
"""Benchmark: attention forward + backward TFLOPS on one GB300 (or N replicas).

One step = the whole hot path over one batch of synthetic input: the forward
(work list, fused attention kernel) and the backward (work list, preprocess
D = rowsum(dO * O), fused dK/dV-stationary kernel with dQ accumulation, dQ
conversion), for the workload named by --workload (default: B=2, H=16,
S=8192, D=128, bf16, no mask).

Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events on
the launching stream; between timed steps a 512 MiB buffer is written to flush
L2 (outside the events).  Work counted is algorithmic: 4*D FLOPs per unmasked
(query, key) pair per head forward, 10*D backward.

Prints ONE JSON line (rank 0).  --impl reference times the float64 CPU oracle
instead, on a bounded sample of the same workload, on the host cores.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            return d, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def peak_value(peaks, key):
    """Find a peak by key in a possibly nested MEASURED_PEAKS.json."""
    if key in peaks and isinstance(peaks[key], (int, float)):
        return float(peaks[key])
    for v in peaks.values():
        if isinstance(v, dict):
            r = peak_value(v, key)
            if r is not None:
                return r
    return None


def flops_of(wl, bm=None):
    from bwd_flashattention_fwd_sm_gb300 import workloads as W
    pairs = W.unmasked_pairs(wl, bm)
    heads = wl.heads_q
    fwd = 4.0 * wl.head_dim * pairs * heads
    bwd = 10.0 * wl.head_dim * pairs * heads
    return fwd, bwd, pairs


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.gpu_id is not None:
            cmd.insert(1, f"--id={self.gpu_id}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(value, dist, device=None):
    """The largest `value` over all ranks (the job is as slow as its slowest rank)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(work_per_rank_step, world, steps, seconds):
    """Work of all ranks over the slowest rank's time (weak scaling: each rank runs
    the full per-GPU workload)."""
    return world * work_per_rank_step * steps / seconds


def gpu_identity(torch):
    try:
        uuid = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        return uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
    except Exception:
        return os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0] or None


# Steps in each timed window of an end-to-end leg.  The first step's upload and
# the last step's download overlap no computation; over 30 steps they are a
# small share, as in a stream of steps.
E2E_STEPS = 30


def pipelined_e2e(torch, dev, host_in, compute, n_steps, warmup, dist=None):
    """End to end through the public API with host buffers: every step copies its
    inputs (the pinned tensors of `host_in`) to the device, runs `compute` on
    them, which returns the step's output tensors, and copies every output back
    to pinned host memory.  The copies run on their own streams,
    double-buffered: step i's inputs travel while step i-1 computes and step
    i-1's results while step i computes.  Every copy of every step is inside
    the timed region.  Three timed windows of n_steps, after `warmup` (at most
    2) untimed steps; returns (median seconds, the windows' seconds, bytes
    copied back per step).  Each window is the slowest rank's."""
    names = list(host_in)
    stream = torch.cuda.current_stream()
    dev_in = [{n: torch.empty_like(host_in[n], device=dev) for n in names} for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    host_out = [None, None]
    keep = []  # device outputs stay referenced until their copies are done

    def run(k):
        comp_done = [None, None]
        for i in range(k):
            slot = i & 1
            with torch.cuda.stream(s_in):
                if comp_done[slot] is not None:
                    s_in.wait_event(comp_done[slot])  # step i-2 no longer reads this slot
                for n in names:
                    dev_in[slot][n].copy_(host_in[n], non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(s_in)
            stream.wait_event(ready)
            outs = compute(dev_in[slot])
            done = torch.cuda.Event()
            done.record(stream)
            comp_done[slot] = done
            if host_out[slot] is None:
                host_out[slot] = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
            with torch.cuda.stream(s_out):
                s_out.wait_event(done)
                for h, t in zip(host_out[slot], outs):
                    h.copy_(t, non_blocking=True)
            keep.append(outs)

    run(max(1, min(warmup, 2)))
    torch.cuda.synchronize()
    keep.clear()
    # three windows, the median reported: the host copies share the node's host
    # memory and links with other jobs, and one window can catch a transient
    windows = []
    for _ in range(3):
        if dist is not None:
            dist.barrier()
        t0 = time.perf_counter()
        run(n_steps)
        torch.cuda.synchronize()
        windows.append(max_over_ranks(time.perf_counter() - t0, dist, dev))
        keep.clear()
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    return statistics.median(windows), windows, d2h


def run_ours(args, wl, rank, world, dist):
    import ctypes

    import torch

    from bwd_flashattention_fwd_sm_gb300 import BlockMask, SeqLens, attn_bwd, attn_fwd, get_status, make_params
    from bwd_flashattention_fwd_sm_gb300 import _lib
    from bwd_flashattention_fwd_sm_gb300 import workloads as W

    lib = _lib.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = W.make_inputs(wl)
    bm = inp.get("block_mask")
    fwd_flops, bwd_flops, pairs = flops_of(wl, bm)
    kw = {"scale": wl.scale}
    if wl.mask == "causal":
        kw["causal"] = True
    if bm is not None:
        kw["block_mask"] = BlockMask.from_csr(bm, device=dev)
    if wl.varlen:
        kw["seqlens"] = SeqLens(inp["cu_seqlens"], device=dev)
        kw["seqlen"] = wl.seqlen
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    # Workspaces allocated once; every call reuses them.
    o, lse = attn_fwd(q, k, v, **kw)
    p = make_params(q, k, **kw)
    ws_f = torch.empty(max(1, lib.attn_fwd_workspace_size(ctypes.byref(p))), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(max(1, lib.attn_bwd_workspace_size(ctypes.byref(p))), dtype=torch.uint8, device=dev)

    det = bool(getattr(args, "deterministic", False))  # attn_bwd_deterministic

    def step():
        o, lse = attn_fwd(q, k, v, workspace=ws_f, **kw)
        dq, dk, dv = attn_bwd(q, k, v, o, do, lse, workspace=ws_b, deterministic=det, **kw)
        return o, lse, dq, dk, dv

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    ev = lambda: torch.cuda.Event(enable_timing=True)
    step_ev = [(ev(), ev()) for _ in range(args.steps)]
    fwd_ev = [(ev(), ev()) for _ in range(args.steps)]
    bwd_ev = [(ev(), ev()) for _ in range(args.steps)]
    pre_ev = [(ev(), ev()) for _ in range(args.steps)]
    cvt_ev = [(ev(), ev()) for _ in range(args.steps)]
    # torch creates the CUDA event behind an Event on its first record: record
    # each once so that the library's timing hook receives real handles.
    for pair in fwd_ev + bwd_ev + pre_ev + cvt_ev:
        for e in pair:
            e.record(stream)
    torch.cuda.synchronize()
    clocks = ClockSampler(gpu_identity(torch)) if rank == 0 else None
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
        time.sleep(0.3)
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        lib.attn_set_timing_events(0, ctypes.c_void_p(fwd_ev[i][0].cuda_event), ctypes.c_void_p(fwd_ev[i][1].cuda_event))
        lib.attn_set_timing_events(1, ctypes.c_void_p(bwd_ev[i][0].cuda_event), ctypes.c_void_p(bwd_ev[i][1].cuda_event))
        lib.attn_set_timing_events(2, ctypes.c_void_p(pre_ev[i][0].cuda_event), ctypes.c_void_p(pre_ev[i][1].cuda_event))
        lib.attn_set_timing_events(3, ctypes.c_void_p(cvt_ev[i][0].cuda_event), ctypes.c_void_p(cvt_ev[i][1].cuda_event))
        step_ev[i][0].record(stream)
        step()
        step_ev[i][1].record(stream)
    for which in range(4):
        lib.attn_set_timing_events(which, None, None)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    status = get_status()
    if status != 0:
        raise RuntimeError(f"device status word set during the benchmark: {status}")

    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    fwd_ms = [a.elapsed_time(b) for a, b in fwd_ev]
    bwd_ms = [a.elapsed_time(b) for a, b in bwd_ev]
    pre_ms = [a.elapsed_time(b) for a, b in pre_ev]
    cvt_ms = [a.elapsed_time(b) for a, b in cvt_ev]
    total_ms = max_over_ranks(sum(step_ms), dist, dev)
    ms_per_step = total_ms / args.steps
    step_flops = fwd_flops + bwd_flops
    value = whole_job_rate(step_flops, world, args.steps, total_ms * 1e-3) / 1e12

    # End to end through the public API with host buffers: every step copies its
    # inputs in from pinned host memory and its results back out.  The copies
    # run on their own streams, double-buffered, so step i's inputs travel
    # while step i-1 computes and step i-1's results travel while step i
    # computes, as an input pipeline would; every copy of every step is inside
    # the timed region.
    names_in = ("q", "k", "v", "do")
    host_in = {n: inp[n].pin_memory() for n in names_in}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())

    def compute(d):
        o_, lse_ = attn_fwd(d["q"], d["k"], d["v"], workspace=ws_f, **kw)
        dq_, dk_, dv_ = attn_bwd(d["q"], d["k"], d["v"], o_, d["do"], lse_, workspace=ws_b, deterministic=det, **kw)
        return o_, lse_, dq_, dk_, dv_

    e2e_steps = E2E_STEPS
    e2e_s, windows, d2h = pipelined_e2e(torch, dev, host_in, compute, e2e_steps, args.warmup, dist)
    keep_gpu_samples(wl, step())
    e2e_value = whole_job_rate(step_flops, world, e2e_steps, e2e_s) / 1e12

    peaks, peak_src = load_peaks()
    peak = peak_value(peaks, "bf16_tflops") or FALLBACK_PEAKS["bf16_tflops"]
    bwd_avg = sum(bwd_ms) / len(bwd_ms)
    fwd_avg = sum(fwd_ms) / len(fwd_ms)
    achieved = bwd_flops / (bwd_avg * 1e-3) / 1e12
    fwd_ach = fwd_flops / (fwd_avg * 1e-3) / 1e12
    traffic = None
    prof = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(prof):
        try:
            with open(prof) as f:
                t = json.load(f)
            if not det and t.get("workload") == wl.name and t.get("kernel_build") == kernel_build_id():
                traffic = t.get("bwd_main_bytes")
        except Exception:
            traffic = None
    # forward: work list, main kernel; backward: work list, preprocess, main
    # kernel, dQ conversion (deterministic: a second work list and the dQ pass
    # instead of the conversion); block-sparse: the mask transpose
    launches_per_step = 2 + (5 if det else 4) + (1 if wl.mask == "block" else 0)
    # the backward's two HBM-bound kernels, against the HBM copy bandwidth
    hbm = peak_value(peaks, "hbm_gbs") or FALLBACK_PEAKS["hbm_gbs"]
    rows = (int(inp["cu_seqlens"][-1]) if wl.varlen else wl.batch * wl.seqlen) * wl.heads_q
    esz = 2 if wl.dtype == "bf16" else 4
    aux = {}
    # (the deterministic backward has no float32 accumulator: no zero fill, no conversion)
    legs = [("bwd_preprocess", pre_ms, 2 * wl.head_dim * esz + 4 + (0 if det else 4 * wl.head_dim))]
    if not det:
        legs.append(("dq_convert", cvt_ms, 4 * wl.head_dim + wl.head_dim * esz))
    for name, times, per_row in legs:
        t = sum(times) / len(times)
        gbs = rows * per_row / (t * 1e-3) / 1e9
        aux[name] = {"ms": round(t, 4), "bytes": rows * per_row, "gbs": round(gbs, 1),
                     "frac_of_hbm": round(gbs / hbm, 4), "bound": "hbm"}

    line = {
        "metric": "attention fwd+bwd TFLOPS (bf16, D=128, S=8192) and % of GB300 BF16 tensor peak",
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if wl.dtype == "bf16" else "f32",
        "data": "synthetic: Q,K,V,dO iid N(0,1) from a fixed seed, rounded to bf16",
        "config": {
            "workload": wl.name + ("_deterministic" if det else ""),
            "batch": wl.batch, "heads_q": wl.heads_q, "heads_kv": wl.heads_kv, "seq_len": wl.seqlen,
            "head_dim": wl.head_dim, "mask": wl.mask, "varlen": wl.varlen,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": "512 MiB L2 flush written between timed steps (outside the step events)",
            "fwd_flops": fwd_flops, "bwd_flops": bwd_flops,
        },
        "fwd_ms": round(fwd_avg, 4), "bwd_ms": round(bwd_avg, 4),
        "fwd_tflops": round(fwd_ach, 2), "bwd_tflops": round(achieved, 2),
        "fwd_frac_of_peak": round(fwd_ach / peak, 4), "bwd_frac_of_peak": round(achieved / peak, 4),
        "roofline": {
            "kernel": ("backward main without dQ + query-stationary dQ pass (attn_bwd_deterministic)" if det else
                       "backward main (dK/dV-stationary, dQ accumulation)"),
            "bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4), "traffic": traffic,
            "peak_source": f"{peak_src} bf16 dense" + (" (MEASURED_PEAKS.json)" if peak_src == "measured" else
                                                        " (no MEASURED_PEAKS.json: 1.9 PFLOP/s burst)"),
        },
        "aux": aux,
        "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "windows_tflops": [round(step_flops * world * e2e_steps / w / 1e12, 1) for w in windows],
                "copies": "pinned host buffers; H2D and D2H on their own streams, double-buffered, "
                          "overlapping the neighbouring steps' kernels"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    return line


# The sources that decide what the backward main kernel reads and writes: its
# own code, the work-list order, the launch and tensor-map setup, and every
# header.  A change elsewhere (the forward, FP8, LayerNorm kernels) leaves its
# DRAM counters valid.
TRAFFIC_SOURCES = ("tc_bwd.cu", "sched.cu", "api.cu", "tma_host.cu")


def kernel_build_id():
    """Hash of the backward main kernel's sources' contents (no paths, so it is
    the same wherever the repository sits); profiles/traffic.json records the id
    of the sources its counters were taken on."""
    import hashlib
    h = hashlib.sha256()
    for d in (os.path.join(ROOT, "bwd_flashattention_fwd_sm_gb300", "csrc"), os.path.join(ROOT, "include")):
        for name in sorted(os.listdir(d)):
            if name in TRAFFIC_SOURCES or name.endswith((".cuh", ".h")):
                h.update(name.encode())
                with open(os.path.join(d, name), "rb") as f:
                    h.update(f.read())
    return h.hexdigest()[:16]


def cpu_model():
    """The host CPU's model name (lscpu's "Model name", else /proc/cpuinfo), or None."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return None


# The device results of the benchmarked workload's first query heads (sequence
# 0 or all packed sequences), kept on the host for cpu_baseline to compare with
# the oracle it runs on the same heads.
_GPU_SAMPLES = {}
SAMPLE_HEADS = 4


def keep_gpu_samples(wl, outs):
    o, lse, dq, dk, dv = outs
    _GPU_SAMPLES.clear()
    G = wl.heads_q // wl.heads_kv
    for h in range(min(SAMPLE_HEADS, wl.heads_q)):
        if wl.varlen:
            sel = lambda t, j: t[:, j:j + 1]
            lse_h = lse[h]
        else:
            sel = lambda t, j: t[0:1, j:j + 1]
            lse_h = lse[0, h]
        d = {"o": sel(o, h), "lse": lse_h, "dq": sel(dq, h)}
        if G == 1:  # with GQA a KV head's dK, dV sum its whole group
            d["dk"], d["dv"] = sel(dk, h), sel(dv, h)
        _GPU_SAMPLES[h] = {n: t.double().cpu().numpy() for n, t in d.items()}


def half_ulp_bf16(x):
    """Half a bfloat16 unit in the last place of each |x| (0 at 0)."""
    import numpy as np
    _, e = np.frexp(np.abs(x))
    return np.where(x == 0, 0.0, np.ldexp(1.0, e - 9))


def sample_parity(wl, refs):
    """max-abs and rel-L2 of the kept device results against the oracle's, per
    tensor over the sampled heads, and whether every element is within the GPU
    tests' bound (bf16: 2e-2 plus half a bf16 ulp of the oracle, rel-L2 1e-2,
    LSE 2e-2; float32: 1e-3)."""
    import numpy as np
    out, ok = {}, True
    for name in ("o", "lse", "dq", "dk", "dv"):
        got = [(_GPU_SAMPLES[h][name], r[name]) for h, r in refs.items() if h in _GPU_SAMPLES and name in _GPU_SAMPLES[h]]
        if not got:
            continue
        g = np.concatenate([a.ravel() for a, _ in got])
        r = np.concatenate([b.ravel() for _, b in got])
        fin = np.isfinite(r)  # fully masked rows: LSE -inf on both sides
        err = np.abs(g[fin] - r[fin])
        rl2 = float(np.linalg.norm(g[fin] - r[fin]) / max(np.linalg.norm(r[fin]), 1e-300))
        if name == "lse":
            good = bool(np.all(err <= 2e-2)) and bool(np.array_equal(np.isfinite(g), fin))
        elif wl.dtype == "bf16":
            good = bool(np.all(err <= 2e-2 + half_ulp_bf16(r[fin]))) and rl2 <= 1e-2
        else:
            good = bool(np.all(err <= 1e-3))
        ok &= good
        out[name] = {"max_abs": float(err.max()) if err.size else 0.0, "rel_l2": rl2}
    out["within_test_bound"] = ok
    out["heads"] = sorted(h for h in refs if h in _GPU_SAMPLES)
    return out


def cpu_baseline(wl, budget_s=20.0, rank=0):
    """The float64 oracle on a bounded sample of the workload: whole heads at full
    length.  When the benchmark kept the device results of those heads, their
    errors against the oracle are reported too (outside the timed region)."""
    import oracle
    from bwd_flashattention_fwd_sm_gb300 import workloads as W

    inp = W.make_inputs(wl)
    cores = os.cpu_count() or 1
    kw = {"scale": wl.scale}
    if wl.mask == "causal":
        kw["causal"] = True
    if wl.mask == "block":
        kw["block_mask"] = inp["block_mask"]
    if wl.varlen:
        cu = inp["cu_seqlens"]
        sel = lambda t, h: t[:, h:h + 1]
        kw["cu_seqlens"] = cu
    else:
        sel = lambda t, h: t[0:1, h:h + 1]
    fwd_flops, bwd_flops, pairs = flops_of(wl, inp.get("block_mask"))
    per_head = (fwd_flops + bwd_flops) / wl.heads_q / (1 if wl.varlen else wl.batch)
    heads_done, flops_done = 0, 0.0
    refs = {}
    t0 = time.perf_counter()
    while True:
        h = heads_done % wl.heads_q
        G = wl.heads_q // wl.heads_kv
        q, do = (sel(inp[n], h).double().numpy() for n in ("q", "do"))
        k, v = (sel(inp[n], h // G).double().numpy() for n in ("k", "v"))
        o_r, lse_r = oracle.attn_fwd(q, k, v, **kw)
        dq_r, dk_r, dv_r = oracle.attn_bwd(q, k, v, do, **kw)
        if h in _GPU_SAMPLES and h not in refs:
            refs[h] = {"o": o_r, "lse": lse_r[0] if wl.varlen else lse_r[0, 0], "dq": dq_r, "dk": dk_r, "dv": dv_r}
        heads_done += 1
        flops_done += per_head
        if time.perf_counter() - t0 >= budget_s * 0.5 or heads_done >= SAMPLE_HEADS:
            break
    dt = time.perf_counter() - t0
    res = {"value": flops_done / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "cpu_model": cpu_model(),
           "kind": "oracle",
           "sample": f"{heads_done} head(s) of {wl.name} at full length (fwd+bwd, float64), {dt:.1f} s",
           "seconds": round(dt, 2), "heads": heads_done}
    if refs:
        res["parity"] = sample_parity(wl, refs)
    return res


def run_reference(args, wl):
    """Reference arm: the float64 oracle as it stands, on the host cores."""
    fwd_flops, bwd_flops, _ = flops_of(wl)
    per_step = []
    base = None
    for i in range(args.warmup + args.steps):
        r = cpu_baseline(wl, budget_s=6.0)
        if i >= args.warmup:
            per_step.append(r)
        base = r
    value = statistics.mean(r["value"] for r in per_step)
    line = {
        "metric": "attention fwd+bwd TFLOPS (bf16, D=128, S=8192) and % of GB300 BF16 tensor peak",
        "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": statistics.mean(r["seconds"] for r in per_step) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: Q,K,V,dO iid N(0,1) from a fixed seed, rounded to bf16",
        "config": {"workload": wl.name, "batch": wl.batch, "heads_q": wl.heads_q, "heads_kv": wl.heads_kv,
                   "seq_len": wl.seqlen, "head_dim": wl.head_dim, "mask": wl.mask,
                   "sample": "each step: whole heads at full length, bounded to a few seconds"},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": base["cores"],
                         "cpu_model": base["cpu_model"], "kind": "oracle", "sample": base["sample"],
                         "seconds_per_step": statistics.mean(r["seconds"] for r in per_step),
                         "heads_per_step": base["heads"]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


LN_ROWS, LN_COLS = 16384, 4096  # 2 x 8192 tokens of a 4096-wide residual stream, bf16


def run_ln(args):
    """Fused residual add + LayerNorm, bf16 [16384, 4096]: HBM GB/s of one call.

    Each call reads x and the residual and writes y and h (8 bytes per element;
    gamma and beta, 32 KB, stay in L2).  The four tensors (512 MiB) exceed L2, so
    no flush is needed between calls."""
    import torch

    from bwd_flashattention_fwd_sm_gb300 import layernorm_residual

    dev = torch.device("cuda", torch.cuda.current_device())
    g = torch.Generator().manual_seed(21)
    x = (torch.randn(LN_ROWS, LN_COLS, generator=g) * 2 + 0.5).to(torch.bfloat16).to(dev)
    r = torch.randn(LN_ROWS, LN_COLS, generator=g).to(torch.bfloat16).to(dev)
    gm = (torch.randn(LN_COLS, generator=g) * 0.5 + 1).to(dev)
    bt = (torch.randn(LN_COLS, generator=g) * 0.1).to(dev)
    for _ in range(args.warmup):
        layernorm_residual(x, r, gm, bt)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(gpu_identity(torch))
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    for a, b in ev:
        a.record()
        layernorm_residual(x, r, gm, bt)
        b.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = [a.elapsed_time(b) for a, b in ev]
    bytes_per_call = 8.0 * LN_ROWS * LN_COLS
    gbs = bytes_per_call * args.steps / (sum(ms) * 1e-3) / 1e9
    # end to end: host tensors in pinned memory, copied in and out every call
    host_in = {"x": x.cpu().pin_memory(), "r": r.cpu().pin_memory()}
    e2e_steps = E2E_STEPS
    e2e_s, _, _ = pipelined_e2e(torch, dev, host_in, lambda d: layernorm_residual(d["x"], d["r"], gm, bt), e2e_steps,
                                args.warmup)
    e2e = bytes_per_call * e2e_steps / e2e_s / 1e9
    peaks, src = load_peaks()
    peak = peak_value(peaks, "hbm_gbs") or FALLBACK_PEAKS["hbm_gbs"]
    line = {
        "metric": "fused residual add + LayerNorm HBM throughput", "value": round(gbs, 1), "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sum(ms) / len(ms), 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: x ~ N(0.5, 2), residual ~ N(0, 1), gamma ~ N(1, 0.5), beta ~ N(0, 0.1), fixed seed",
        "config": {"workload": f"ln_residual_{LN_ROWS}x{LN_COLS}_bf16", "rows": LN_ROWS, "cols": LN_COLS,
                   "l2": "inputs and outputs (512 MiB) larger than L2; no flush"},
        "roofline": {"kernel": "k_ln_residual", "bound": "hbm", "achieved": round(gbs, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(gbs / peak, 4), "traffic": None,
                     "peak_source": f"{src} HBM copy bandwidth"},
        "e2e": {"value": round(e2e, 1), "unit": "GB/s", "h2d_bytes_per_step": 4 * LN_ROWS * LN_COLS,
                "d2h_bytes_per_step": 4 * LN_ROWS * LN_COLS, "steps": e2e_steps},
        "gpu_launches": args.steps,
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        import oracle.ln as oln
        rows = 256
        t0 = time.time()
        oln.ln_residual(x[:rows].double().cpu().numpy(), r[:rows].double().cpu().numpy(), gm.double().cpu().numpy(),
                        bt.double().cpu().numpy())
        sec = time.time() - t0
        line["cpu_baseline"] = {"value": round(8.0 * rows * LN_COLS / sec / 1e9, 4), "unit": "GB/s", "cores": 1,
                                "kind": "oracle", "sample": f"{rows} rows of the workload, float64 numpy",
                                "seconds": round(sec, 3)}
    return line


def run_fp8(args, wl):
    """FP8 (e4m3) forward: one step = per-tile quantisation of Q, K, V plus the
    FP8 forward kernel, over the workload's batch (fixed length).  `value` counts
    the forward's algorithmic FLOPs (4 D per unmasked pair per head) over the
    whole step; the roofline covers the forward kernel alone, against the
    measured bf16 dense peak times the nominal FP8 / bf16 ratio (4.5 / 2.25)."""
    import ctypes

    import torch

    from bwd_flashattention_fwd_sm_gb300 import BlockMask, attn_fwd_fp8, get_status, quantize_fp8
    from bwd_flashattention_fwd_sm_gb300 import _lib
    from bwd_flashattention_fwd_sm_gb300 import workloads as W

    if wl.varlen or wl.head_dim != 128 or wl.dtype != "bf16":
        raise SystemExit("--fp8 takes fixed-length bf16 workloads with head_dim 128")
    lib = _lib.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = W.make_inputs(wl)
    bm = inp.get("block_mask")
    fwd_flops, _, pairs = flops_of(wl, bm)
    kw = {"scale": wl.scale, "causal": wl.mask == "causal"}
    if bm is not None:
        kw["block_mask"] = BlockMask.from_csr(bm, device=dev)
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    f = quantize_fp8(q, k, v)
    o, lse = attn_fwd_fp8(f, **kw)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=dev)

    def step():
        quantize_fp8(q, k, v, out=f)
        return attn_fwd_fp8(f, workspace=ws, out=o, **kw)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    step_ev = [(ev(), ev()) for _ in range(args.steps)]
    fwd_ev = [(ev(), ev()) for _ in range(args.steps)]
    quant_ev = [(ev(), ev()) for _ in range(args.steps)]
    for pair in fwd_ev:
        for e in pair:
            e.record(stream)
    torch.cuda.synchronize()
    clocks = ClockSampler(gpu_identity(torch))
    clocks.start()
    time.sleep(0.3)
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        lib.attn_set_timing_events(0, ctypes.c_void_p(fwd_ev[i][0].cuda_event), ctypes.c_void_p(fwd_ev[i][1].cuda_event))
        step_ev[i][0].record(stream)
        quant_ev[i][0].record(stream)  # the step, as step() runs it, with the quantiser's own events
        quantize_fp8(q, k, v, out=f)
        quant_ev[i][1].record(stream)
        attn_fwd_fp8(f, workspace=ws, out=o, **kw)
        step_ev[i][1].record(stream)
    lib.attn_set_timing_events(0, None, None)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if get_status() != 0:
        raise RuntimeError("device status word set during the benchmark")
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    fwd_ms = [a.elapsed_time(b) for a, b in fwd_ev]
    ms_per_step = sum(step_ms) / len(step_ms)
    fwd_avg = sum(fwd_ms) / len(fwd_ms)
    value = fwd_flops / (ms_per_step * 1e-3) / 1e12
    achieved = fwd_flops / (fwd_avg * 1e-3) / 1e12
    quant_ms = sum(a.elapsed_time(b) for a, b in quant_ev) / len(quant_ev)  # the quantisation kernel
    elems = (wl.heads_q + 2 * wl.heads_kv) * wl.batch * wl.seqlen * wl.head_dim
    quant_bytes = 3 * elems  # 2 bytes read and 1 written per element

    # end to end: bf16 inputs from pinned host memory, O and LSE back, every step
    host_in = {"q": q.cpu().pin_memory(), "k": k.cpu().pin_memory(), "v": v.cpu().pin_memory()}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())

    def compute(d):  # the quantised operands f are rewritten in stream order each step
        quantize_fp8(d["q"], d["k"], d["v"], out=f)
        return attn_fwd_fp8(f, workspace=ws, **kw)

    e2e_steps = E2E_STEPS
    e2e_s, _, d2h = pipelined_e2e(torch, dev, host_in, compute, e2e_steps, args.warmup)
    e2e = fwd_flops * e2e_steps / e2e_s / 1e12

    peaks, src = load_peaks()
    bf16_peak = peak_value(peaks, "bf16_tflops") or FALLBACK_PEAKS["bf16_tflops"]
    peak = 2.0 * bf16_peak
    hbm = peak_value(peaks, "hbm_gbs") or FALLBACK_PEAKS["hbm_gbs"]
    qgbs = quant_bytes / (quant_ms * 1e-3) / 1e9
    line = {
        "metric": "attention forward TFLOPS with e4m3 operands (D=128, S=8192) and % of GB300 FP8 tensor peak",
        "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3",
        "data": "synthetic: Q,K,V iid N(0,1) from a fixed seed, rounded to bf16, quantised per 128-row tile",
        "config": {"workload": wl.name + "_fp8", "batch": wl.batch, "heads_q": wl.heads_q, "heads_kv": wl.heads_kv,
                   "seq_len": wl.seqlen, "head_dim": wl.head_dim, "mask": wl.mask,
                   "step": "attn_quantize_fp8 + attn_fwd_fp8",
                   "l2": "512 MiB L2 flush written between timed steps (outside the step events)",
                   "fwd_flops": fwd_flops},
        "fwd_ms": round(fwd_avg, 4), "fwd_tflops": round(achieved, 2),
        "roofline": {"kernel": "FP8 forward (k_tc_fwd, e4m3 operands)", "bound": "tensor",
                     "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": None,
                     "peak_source": f"{src} bf16 dense x 2 (nominal FP8 / bf16 ratio 4.5 / 2.25 PFLOP/s)"},
        "aux": {"quantize": {"ms": round(quant_ms, 4), "bytes": quant_bytes, "gbs": round(qgbs, 1),
                             "frac_of_hbm": round(qgbs / hbm, 4), "bound": "hbm",
                             "note": "events around the quantisation kernel (one launch for Q, K and V)"}},
        "e2e": {"value": round(e2e, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps},
        "gpu_launches": 3 * args.steps,
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        import oracle
        from oracle import fp8 as ofp8
        t0 = time.perf_counter()
        sl = (slice(0, 1), slice(0, 1))
        deq = [ofp8.dequantize(*ofp8.quantize_tiles(inp[n][sl].float().numpy())) for n in ("q", "k", "v")]
        oracle.attn_fwd(*deq, scale=wl.scale, causal=wl.mask == "causal", block_mask=bm)
        sec = time.perf_counter() - t0
        per_head = fwd_flops / wl.heads_q / wl.batch
        line["cpu_baseline"] = {"value": per_head / sec / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count() or 1,
                                "kind": "oracle",
                                "sample": f"1 head of {wl.name} at full length: quantise + float64 forward",
                                "seconds": round(sec, 2)}
    return line


def run_d256(args):
    """Head dim 256: the forward and backward step on d256_dense_s8192 (B=2, H=16,
    S=8192), both passes on the tensor cores, measured like the main step."""
    from bwd_flashattention_fwd_sm_gb300 import workloads as W
    wl = W.WORKLOADS["d256_dense_s8192"]
    line = run_ours(args, wl, 0, 1, None)
    line["metric"] = "attention fwd+bwd TFLOPS at head dim 256 (bf16, S=8192) and % of GB300 BF16 tensor peak"
    line["roofline"]["kernel"] = "head-dim-256 backward (k_tc_bwd256: each key tile once per head-dim half)"
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl)
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="h0_dense_s8192")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ln", action="store_true",
                    help="measure the fused residual add + LayerNorm instead of attention")
    ap.add_argument("--fp8", action="store_true",
                    help="measure the FP8 (e4m3) forward (quantisation + forward) on --workload")
    ap.add_argument("--d256", action="store_true",
                    help="measure head dim 256: forward and backward at B=2, H=16, S=8192")
    ap.add_argument("--deterministic", action="store_true",
                    help="run the backward as attn_bwd_deterministic (fixed dQ summation order)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.ln:
        if int(os.environ.get("RANK", "0")) == 0 and args.impl == "ours":
            print(json.dumps(run_ln(args)), flush=True)
        return 0
    if args.d256:
        if int(os.environ.get("RANK", "0")) == 0 and args.impl == "ours":
            print(json.dumps(run_d256(args)), flush=True)
        return 0

    from bwd_flashattention_fwd_sm_gb300 import workloads as W
    wl = W.WORKLOADS[args.workload]
    if args.fp8:
        if int(os.environ.get("RANK", "0")) == 0 and args.impl == "ours":
            print(json.dumps(run_fp8(args, wl)), flush=True)
        return 0

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, wl)), flush=True)
        return 0

    import torch
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        dist_mod.init_process_group("nccl")
        dist = dist_mod
    line = run_ours(args, wl, rank, world, dist)
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(wl)
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
