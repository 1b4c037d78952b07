#!/usr/bin/env python
"""Benchmark of the GB300 KDA chunked forward; prints one JSON line.

A step is one full forward through the C ABI (kda_fwd: chunk planner +
intra-chunk kernel + scan kernel) over the headline workload (B=4, H=32, T=8192, K=V=128, bf16 I/O, fp32
state), inputs resident in HBM.  The inputs (1.6 GB) are larger than L2, so
no flush is done between steps.  Every step has its own CUDA events; the line
reports the median (the value), p10 and p90.  After the timed region a
labelled clock-only window of untimed steps (about 0.5 s) gives the clock
sampler several samples however short the timed region is.  The line also
carries both HBM fractions of the step (two-stage algorithmic bytes and the
strict single-pass I/O), the mid, varlen and long workloads timed in the same
run (``other_workloads``; --no-configs skips them) and, from the CPU-baseline
leg, the smoke-size parity figures against the fp64 oracle.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                  [--path fwd|bwd_dh] [--workload NAME]

--path bwd_dh times the reverse state scan (kda_bwd_dh) instead, on the
forward's workspace of the same inputs, and prints its own line.

--impl reference times the fp64 CPU oracle (the only reference this method
has) on a bounded sample of the same workload on the host cores.  Under
torchrun each rank runs an independent replica (the path shards into
independent (sequence, head) units; no collective on the data path).
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

METRIC = "KDA fwd tokens/s (B=4,H=32,T=8192,K=V=128 bf16); % of HBM/TC roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ----------------------------------------------------------------------------- helpers
from chunked_gated_delta_gb300.dist import barrier, max_over_ranks, rank_info  # noqa: E402


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def bytes_per_token_head(K, V, C=64):
    """Algorithmic HBM bytes per token-head of each kernel (two-stage chunked form)."""
    intra = (2 * K * 2 + V * 2 + K * 4 + 2) + (3 * K * 2 + V * 2 + C * 2 + K * 4 / C)
    scan = (3 * K * 2 + C * 2 + V * 2 + K * 4 / C) + V * 2
    return intra, scan


def flops_per_token_head(K, V, C=64):
    """Chunked-form flops per token-head (Aqk, A, w, u; WH, qg@h, kg^T v'; Aqk@v')."""
    per_chunk = 2 * C * C * K * 3 + 2 * C * C * V + 3 * 2 * C * K * V + 2 * C * C * V
    return per_chunk / C


# headers every kernel translation unit compiles in (PTX wrappers, layouts)
KERNEL_HEADERS = ("ptx.cuh", "common.cuh", "internal.h", "chunk_math.cuh")


def code_text(src):
    """C / CUDA source without its comments and blank lines (string and
    character literals kept as written), so that a change to comments alone
    leaves a kernel's key unchanged and any change to code changes it."""
    out, i, n = [], 0, len(src)
    while i < n:
        ch = src[i]
        if ch in "\"'":
            j = i + 1
            while j < n and src[j] != ch:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(ch)
            i += 1
    lines = (ln.rstrip() for ln in "".join(out).splitlines())
    return "\n".join(ln for ln in lines if ln)


def source_sha(path):
    """sha256 prefix of a kernel source together with the headers it includes,
    over their code (comments and blank lines left out)."""
    h = hashlib.sha256()
    for p in [path] + [os.path.join(os.path.dirname(path), n) for n in KERNEL_HEADERS]:
        with open(p, encoding="utf-8") as f:
            h.update(code_text(f.read()).encode("utf-8"))
    return h.hexdigest()[:16]


def ncu_traffic(kernel_name, src_file, workload):
    """Per-launch DRAM bytes of a kernel from the committed ncu summary, if the
    kernel source is unchanged since the capture (else None)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = source_sha(src_file)
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kv = dict(tok.split("=", 1) for tok in line.split() if "=" in tok)
            if (kv.get("kernel") == kernel_name and kv.get("workload") == workload
                    and kv.get("source_sha") == sha):
                try:
                    return float(kv["dram_bytes_per_launch"])
                except (KeyError, ValueError):
                    return None
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 25 ms while running.
    Each line is stamped with the host clock on arrival.  mark_start() /
    mark_end() bracket the timed region; mark_window() brackets a clock-only
    window of back-to-back untimed steps run after it (a timed region of a
    few milliseconds can fall between two samples).  stop() waits until a
    sample stamped after the last mark has arrived, then reports the samples
    inside the timed region and inside the window separately."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    SLACK = 0.03  # a sample arriving this soon after a mark was taken before it

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None
        self.t0 = self.t1 = self.w0 = self.w1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "25"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def mark_start(self):
        self.t0 = time.monotonic()

    def mark_end(self):
        self.t1 = time.monotonic()

    def mark_window(self, w0, w1):
        self.w0, self.w1 = w0, w1

    @staticmethod
    def parse(lines):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return sm, smax, reasons

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "samples": 0, "reasons": ["nvidia-smi unavailable"]}
        last = max([t for t in (self.t1, self.w1) if t is not None], default=None)
        deadline = time.monotonic() + 2.0
        while last is not None and time.monotonic() < deadline and not any(t > last + self.SLACK
                                                                            for t, _ in self.lines):
            time.sleep(0.01)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        lines = list(self.lines)
        region = [x for x in lines if self.t0 is not None and self.t0 <= x[0] <= self.t1 + self.SLACK]
        window = [x for x in lines if self.w0 is not None and self.w0 <= x[0] <= self.w1 + self.SLACK]
        after = [x for x in lines if self.t1 is not None and x[0] > self.t1 + self.SLACK][:1]
        sm_r, smax_r, why_r = self.parse(region)
        sm_w, smax_w, why_w = self.parse(window)
        sm_a, smax_a, why_a = self.parse(after)
        if sm_r:
            used, which = sm_r, "timed region"
        elif sm_w:
            used, which = sm_w, "clock window (untimed back-to-back steps right after the timed region)"
        else:
            used, which = sm_a, "first sample after the timed region"
        smax = smax_r + smax_w + smax_a
        return {"sm_mhz": statistics.median(used) if used else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(used), "window": which,
                "samples_in_region": len(sm_r), "sm_mhz_in_region": statistics.median(sm_r) if sm_r else None,
                "samples_clock_window": len(sm_w),
                "sm_mhz_clock_window": statistics.median(sm_w) if sm_w else None,
                "clock_window_s": (self.w1 - self.w0) if self.w0 is not None else None,
                "reasons": sorted(why_r | why_w | why_a)}


def time_steps(step, n, stream):
    """Runs n steps with a CUDA event between consecutive steps on `stream`;
    returns (per-step ms list, first-to-last span ms)."""
    import torch
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    ev[0].record(stream)
    for i in range(n):
        step()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    return [ev[i].elapsed_time(ev[i + 1]) for i in range(n)], ev[0].elapsed_time(ev[-1])


def pct(xs, q):
    """The q-quantile (0..1) of xs by linear interpolation."""
    ys = sorted(xs)
    if not ys:
        return None
    pos = q * (len(ys) - 1)
    lo = int(pos)
    hi = min(lo + 1, len(ys) - 1)
    return ys[lo] + (ys[hi] - ys[lo]) * (pos - lo)


def clock_window(step, ms_per_step, clocks, seconds=0.5):
    """Untimed back-to-back steps for about `seconds` of GPU time, bracketed
    for the clock sampler (outside the timed region)."""
    import torch
    n = max(1, int(seconds * 1e3 / max(ms_per_step, 1e-3)) + 1)
    w0 = time.monotonic()
    for _ in range(n):
        step()
    torch.cuda.synchronize()
    clocks.mark_window(w0, time.monotonic())
    return n


def host_cores():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


# ----------------------------------------------------------------------------- CPU oracle timing
def oracle_sample_rate(x, seconds, cores):
    """Time the fp64 oracle on a bounded sample of (sequence, head) units of the
    workload; returns (tokens/s scaled to whole tokens, description, threads)."""
    import numpy as np
    import oracle
    B, T, H = x["B"], x["T"], x["H"]
    # calibrate with one unit on one thread
    sub = lambda nh: {n: x[n][:1, :, :nh].contiguous() for n in ("q", "k", "v", "g", "beta")}  # noqa: E731
    one = sub(1)
    h0 = None if x["h0"] is None else x["h0"][:1, :1].contiguous()
    t0 = time.perf_counter()
    oracle.recurrent_fwd(one["q"], one["k"], one["v"], one["g"], one["beta"], x["scale"], h0=h0,
                         nthreads=1)
    t1 = time.perf_counter() - t0
    nh = int(max(1, min(H, round(seconds * cores / max(t1, 1e-6)))))
    s = sub(nh)
    h0 = None if x["h0"] is None else x["h0"][:1, :nh].contiguous()
    th = min(cores, nh)
    t0 = time.perf_counter()
    oracle.recurrent_fwd(s["q"], s["k"], s["v"], s["g"], s["beta"], x["scale"], h0=h0, nthreads=th)
    dt = time.perf_counter() - t0
    tokens_equiv = T * nh / H
    desc = (f"fp64 oracle on {nh} of the {B * H} (sequence, head) units (sequence 0, heads 0..{nh - 1}), "
            f"{T} tokens each; rate scaled to whole {H}-head tokens")
    return tokens_equiv / dt, desc, th, dt


# ----------------------------------------------------------------------------- arms
def run_reference(args):
    rank, world, _ = rank_info()
    if rank != 0:
        return 0
    from chunked_gated_delta_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    x = synth.make_inputs(w)
    cores = host_cores()
    bwd = args.path == "bwd_dh"
    gr = synth.make_bwd_inputs(x) if bwd else None
    rates = []
    for i in range(args.warmup + args.steps):
        if bwd:
            r, desc, dt = oracle_bwd_sample_rate(x, gr, args.ref_seconds)
            th = 1
        else:
            r, desc, th, dt = oracle_sample_rate(x, args.ref_seconds, cores)
        if i >= args.warmup:
            rates.append((r, dt))
    value = statistics.median(r for r, _ in rates)
    ms = statistics.median(dt for _, dt in rates) * 1000
    line = {
        "impl": "reference", "metric": BWD_METRIC if bwd else METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {**workload_config(w, x), "path": "bwd_dh"} if bwd else workload_config(w, x),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": th, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w, x):
    return {"workload": f"{w.name}: B={x['B']} H={x['H']} T={x['T']} K={x['K']} V={x['V']} chunk=64",
            "B": x["B"], "T": x["T"], "H": x["H"], "K": x["K"], "V": x["V"], "chunk": 64,
            "l2": "inputs (~1.6 GB) larger than L2 (129 MB); no flush between steps",
            "parallelism": "independent replica per GPU"}


def launches_per_step(lay):
    """Kernel launches of one kda_fwd call for a workspace layout."""
    if lay.stage_count > 1:
        return 1 + 2 * lay.stage_count
    return 3 + (2 if lay.seg_count > 1 else 0)


def strict_bytes_per_token_head(K, V):
    """Bytes per token-head a single-pass forward must move: read q, k, v, g,
    beta once and write o once (the intermediates never leave the chip)."""
    return 2 * K * 2 + V * 2 + K * 4 + 2 + V * 2


def step_roofline(K, V, tokens_heads, state_bytes, ms, hbm, tc):
    """Both HBM bounds of one forward (two-stage algorithmic bytes, and the
    strict single-pass I/O) and the tensor-core time, with the fractions a
    step of `ms` milliseconds reaches."""
    b_intra, b_scan = bytes_per_token_head(K, V)
    two = (b_intra + b_scan) * tokens_heads + state_bytes
    strict = strict_bytes_per_token_head(K, V) * tokens_heads + state_bytes
    flops = flops_per_token_head(K, V) * tokens_heads
    two_ms = two / (hbm * 1e9) * 1e3
    strict_ms = strict / (hbm * 1e9) * 1e3
    return {"bytes": two, "hbm_ms": two_ms, "frac_of_hbm_bound": two_ms / ms,
            "strict_io_bytes": strict, "strict_io_hbm_ms": strict_ms, "frac_of_strict_io_bound": strict_ms / ms,
            "flops": flops, "tc_ms": flops / (tc * 1e12) * 1e3}


def measure_workload(kda, name, dev, steps, hbm, tc):
    """One extra workload's forward timed in the same run (inputs drawn on the
    device, same distributions; its own warm-up): median and p10/p90 per step
    and its roofline fractions."""
    import torch
    from chunked_gated_delta_gb300 import synth
    w = synth.WORKLOADS[name]
    x = synth.make_inputs_on(w, dev)
    B, T, H, K, V, N = x["B"], x["T"], x["H"], x["K"], x["V"], x["N"]
    dims = kda.make_dims(B, T, H, K, V, 0 if x["cu_seqlens"] is None else N)
    ws = kda.new_workspace(dims, dev)
    o = torch.empty((B, T, H, V), dtype=torch.bfloat16, device=dev)
    ht = torch.empty((N, H, K, V), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        kda.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"], cu_seqlens=x["cu_seqlens"],
                workspace=ws, out=o, final_state=ht, stream=stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    if kda.status(ws, stream) != 0:
        raise RuntimeError(f"kernel status on {name}")
    per, _ = time_steps(step, steps, stream)
    med = statistics.median(per)
    tokens = B * T
    hstate = (2 if x["h0"] is not None else 1) * N * H * K * V * 4
    lay = kda.workspace_layout(dims)
    out = {"workload": workload_config(w, x)["workload"], "steps": steps, "ms_per_step": med,
           "ms_p10": pct(per, 0.1), "ms_p90": pct(per, 0.9), "tokens_per_s": tokens / (med / 1e3),
           "launches_per_step": launches_per_step(lay), "plan": plan_name(lay),
           "step_roofline": step_roofline(K, V, tokens * H, hstate, med, hbm, tc)}
    del x, ws, o, ht
    torch.cuda.empty_cache()
    return out


def plan_name(lay):
    if lay.stage_count > 1:
        return f"staged ({lay.stage_count} chunk ranges of {lay.stage_len})"
    if lay.seg_count > 1:
        return f"segmented scan ({lay.seg_count} segments of {lay.seg_len} chunks)"
    return "two-stage (intra kernel, then scan)"


def gpu_parity_small(kda, dev):
    """GPU results of the smoke-size problems whose parity the CPU-baseline
    leg reports: the tiny workload and a two-sequence K = V = 128 problem."""
    import torch
    from chunked_gated_delta_gb300 import synth
    out = {}
    for name, w in (("tiny", synth.WORKLOADS["tiny"]),
                    ("smoke", synth.Workload("smoke", B=2, T=150, H=2, K=128, V=128, seed=7))):
        x = synth.make_inputs(w)
        d = {n: (x[n].to(dev) if isinstance(x[n], torch.Tensor) else x[n]) for n in x}
        o, ht = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"])
        torch.cuda.synchronize(dev)
        out[name] = (x, o.cpu(), ht.cpu())
    return out


def parity_figures(small):
    """Errors of the GPU results against the fp64 oracle (the tolerances the
    tests hold: rel_o, rel_ht <= 5e-3, maxrel_o <= 2e-2)."""
    import numpy as np
    import oracle
    res = {}
    for name, (x, o, ht) in small.items():
        o_ref, ht_ref = oracle.recurrent_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"])
        og = o.double().numpy()
        res[name] = {"rel_o": float(np.linalg.norm(og - o_ref) / np.linalg.norm(o_ref)),
                     "maxrel_o": float(np.max(np.abs(og - o_ref)) / np.max(np.abs(o_ref))),
                     "rel_ht": float(np.linalg.norm(ht.double().numpy() - ht_ref) / np.linalg.norm(ht_ref))}
    return res


def run_gb300(args):
    import torch
    rank, world, local = rank_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    import chunked_gated_delta_gb300 as kda
    from chunked_gated_delta_gb300 import synth
    kda.load_library(build_if_missing=True)

    w = synth.WORKLOADS[args.workload]
    x = synth.make_inputs(w)
    B, T, H, K, V, N = x["B"], x["T"], x["H"], x["K"], x["V"], x["N"]
    d = {n: (x[n].to(dev) if isinstance(x[n], torch.Tensor) else x[n]) for n in x}
    dims = kda.make_dims(B, T, H, K, V, 0 if x["cu_seqlens"] is None else N)
    ws = kda.new_workspace(dims, dev)
    o = torch.empty((B, T, H, V), dtype=torch.bfloat16, device=dev)
    ht = torch.empty((N, H, K, V), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    lib = kda.load_library()
    import ctypes
    P = lambda t: ctypes.c_void_p(0 if t is None else t.data_ptr())  # noqa: E731
    args_c = (P(d["q"]), P(d["k"]), P(d["v"]), P(d["g"]), P(d["beta"]), ctypes.c_float(d["scale"]), P(d["h0"]),
              P(d["cu_seqlens"]), P(o), P(ht), ctypes.byref(dims), P(ws), ctypes.c_size_t(ws.numel()),
              ctypes.c_void_p(stream.cuda_stream))

    fused = args.plan == "fused"
    opts = kda.FwdOpts(0, 0, 0, 0, kda.binding.PLAN_FUSED if fused else kda.binding.PLAN_AUTO)
    args_ex = args_c[:10] + (ctypes.byref(dims), ctypes.byref(opts)) + args_c[11:]

    def step():
        # one full forward through the C ABI (planner, intra-chunk kernel, scan;
        # or planner and the single-pass fused kernel)
        rc = lib.kda_fwd_ex(*args_ex) if fused else lib.kda_fwd(*args_c)
        if rc != 0:
            raise RuntimeError(kda.status_string(rc))

    def split_step(ev_mid):
        kda.fwd_intra(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], dims, ws, stream)
        ev_mid.record(stream)
        kda.fwd_scan(d["scale"], d["h0"], o, ht, dims, ws, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st = kda.status(ws, stream)
    if st != 0:
        raise RuntimeError(f"kernel status {st}")

    # timed region: K full forwards back to back, an event between consecutive steps
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.mark_start()
    per_step, span_ms = time_steps(step, args.steps, stream)
    clocks.mark_end()
    barrier(world)
    med = statistics.median(per_step)
    # clock-only window: untimed back-to-back steps right after the region
    window_steps = clock_window(step, med, clocks)
    clk = clocks.stop()
    clk["clock_window_steps"] = window_steps
    ms_per_step = max_over_ranks(med, world)
    ms_mean = max_over_ranks(span_ms / args.steps, world)

    # per-kernel split (separate steps with an event between the two kernels)
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    ev0[0].record(stream)
    for i in range(args.steps):
        split_step(ev1[i])
        ev0[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    intra_ms = [ev0[i].elapsed_time(ev1[i]) for i in range(args.steps)]
    scan_ms = [ev1[i].elapsed_time(ev0[i + 1]) for i in range(args.steps)]
    if fused:  # restore the fused path's outputs (the split steps overwrote o / ht)
        step()
        torch.cuda.synchronize(dev)
    tokens = B * T
    value = tokens * world / (ms_per_step / 1e3)

    lay = kda.workspace_layout(dims)
    # roofline of the dominant kernel
    hbm, tc, tc_sus, peak_kind = peaks()
    b_intra, b_scan = bytes_per_token_head(K, V)
    th = tokens * H
    hstate = 2 * N * H * K * V * 4 if x["h0"] is not None else N * H * K * V * 4
    intra_med = statistics.median(intra_ms)
    scan_med = statistics.median(scan_ms)
    if fused:  # one kernel moving the strict single-pass I/O (the planner is microseconds)
        dom, dom_ms, dom_bytes, src = ("kda_fused_kernel", ms_per_step,
                                       strict_bytes_per_token_head(K, V) * th + hstate, "fused.cu")
    elif scan_med >= intra_med:
        dom, dom_ms, dom_bytes, src = "kda_scan_kernel", scan_med, b_scan * th + hstate, "scan.cu"
    else:
        dom, dom_ms, dom_bytes, src = "kda_intra_kernel", intra_med, b_intra * th, "intra.cu"
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    traffic = ncu_traffic(dom, os.path.join(ROOT, "chunked_gated_delta_gb300", "csrc", src), w.name)

    # end to end through the C ABI with host buffers (pinned), copies inside the timed region
    e2e = run_e2e(args, kda, x, dims, stream, dev, world) if (args.e2e_steps > 0 and not fused) else None
    small = gpu_parity_small(kda, dev) if (rank == 0 and not args.no_cpu_baseline) else None
    del ws, o, ht, d
    torch.cuda.empty_cache()
    others = {}
    if args.configs and rank == 0:
        for name in ("mid", "varlen", "long"):
            if name != args.workload:
                others[name] = measure_workload(kda, name, dev, min(args.steps, 50), hbm, tc)

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; shapes and distributions of the KDA forward workloads)",
        "config": workload_config(w, x),
        "timing": {"ms_per_step_median": ms_per_step, "ms_p10": pct(per_step, 0.1), "ms_p90": pct(per_step, 0.9),
                   "ms_per_step_mean": ms_mean, "per_step_events": True,
                   "note": "value = tokens / median per-step time (CUDA events between consecutive steps on the "
                           "launching stream, max over ranks)"},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": traffic, "peak_kind": peak_kind,
                     "algorithmic_bytes_per_launch": dom_bytes, "avg_launch_ms": dom_ms,
                     "launch_ms_statistic": ("median of the timed steps (planner launch included)" if fused
                                             else "median over the split steps")},
        "step_roofline": step_roofline(K, V, th, hstate, ms_per_step, hbm, tc),
        "kernels_ms": {"intra": intra_med, "scan": scan_med, "note": "medians of separate split steps with an "
                       "event between the kernels over every chunk; the timed steps run them back to back"
                       + (f", in {lay.stage_count} chunk ranges of {lay.stage_len} chunks (each range's "
                          "intra kernel beside the previous range's scan)" if lay.stage_count > 1 else "")},
        "plan": "single-pass fused kernel (one CTA per sequence and head)" if fused else plan_name(lay),
        "e2e": e2e,
        # planner + intra + scan (+ map pass and combine when the scan is segmented;
        # planner + one intra and one scan per chunk range when the forward is staged;
        # planner + the fused kernel on the fused plan)
        "gpu_launches": (2 if fused else launches_per_step(lay)) * args.steps,
        "clocks": clk,
    }
    if others:
        line["other_workloads"] = others
    if rank == 0 and not args.no_cpu_baseline:
        r, desc, thr, _ = oracle_sample_rate(x, args.ref_seconds, host_cores())
        line["cpu_baseline"] = {"value": r, "unit": "tokens/s", "cores": thr, "kind": "oracle",
                                "sample": desc}
        line["parity"] = parity_figures(small)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


BWD_METRIC = "KDA reverse state scan (dh, dv2, dh0) tokens/s (B=4,H=32,T=8192,K=V=128 bf16); % of HBM roofline"


def bwd_bytes_per_token_head(K, V, C=64):
    """Algorithmic HBM bytes per token-head of the reverse state scan: reads qg,
    kg, w (workspace), do, dv_in and the chunk decay; writes dv2 and the bf16
    dh checkpoint (K x V per chunk)."""
    return 3 * K * 2 + 2 * V * 2 + K * 4 / C + V * 2 + K * V * 2 / C


def oracle_bwd_sample_rate(x, gr, seconds):
    """Time the fp64 reverse-scan oracle on a bounded sample of (sequence, head)
    units (one thread: it is numpy); returns (tokens/s scaled, description, dt)."""
    from oracle import chunked as oc
    f = lambda t: None if t is None else t.double().numpy()  # noqa: E731
    B, T, H = x["B"], x["T"], x["H"]
    sl = lambda t: None if t is None else t[:1]  # noqa: E731
    args = [f(sl(x[n])) for n in ("q", "k", "v", "g", "beta")]
    do, dvi = f(sl(gr["do"])), f(sl(gr["dv_in"]))
    dht = None if gr["dht"] is None else f(gr["dht"][:1])
    t0 = time.perf_counter()
    oc.chunked_bwd_dh(*args, x["scale"], do, dvi, dht=dht, units=[(0, 0)])
    t1 = time.perf_counter() - t0
    nh = int(max(1, min(H, round(seconds / max(t1, 1e-6)))))
    t0 = time.perf_counter()
    oc.chunked_bwd_dh(*args, x["scale"], do, dvi, dht=dht, units=[(0, h) for h in range(nh)])
    dt = time.perf_counter() - t0
    desc = (f"fp64 chunked reverse-scan oracle (numpy, 1 thread) on {nh} of the {B * H} (sequence, head) "
            f"units (sequence 0, heads 0..{nh - 1}), {T} tokens each; rate scaled to whole {H}-head tokens")
    return T * nh / H / dt, desc, dt


def run_gb300_bwd(args):
    """The reverse state scan (kda_bwd_dh) on the workload: a step is one call
    over all (sequence, head) units, the forward's workspace already filled."""
    import torch
    rank, world, local = rank_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    import chunked_gated_delta_gb300 as kda
    from chunked_gated_delta_gb300 import synth
    kda.load_library(build_if_missing=True)
    w = synth.WORKLOADS[args.workload]
    x = synth.make_inputs(w)
    gr = synth.make_bwd_inputs(x)
    B, T, H, K, V, N = x["B"], x["T"], x["H"], x["K"], x["V"], x["N"]
    d = {n: (x[n].to(dev) if isinstance(x[n], torch.Tensor) else x[n]) for n in x}
    g = {n: (t.to(dev) if t is not None else None) for n, t in gr.items()}
    dims = kda.make_dims(B, T, H, K, V, 0 if x["cu_seqlens"] is None else N)
    ws = kda.new_workspace(dims, dev)
    stream = torch.cuda.current_stream(dev)
    kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"], cu_seqlens=d["cu_seqlens"],
            output_final_state=False, workspace=ws, stream=stream)
    lay = kda.workspace_layout(dims)
    dhck = torch.empty((lay.max_chunks, H, K, V), dtype=torch.bfloat16, device=dev)
    dv2 = torch.empty((B, T, H, V), dtype=torch.bfloat16, device=dev)
    dh0 = torch.empty((N, H, K, V), dtype=torch.float32, device=dev)
    lib = kda.load_library()
    import ctypes
    P = lambda t: ctypes.c_void_p(0 if t is None else t.data_ptr())  # noqa: E731

    def step():
        rc = lib.kda_bwd_dh(ctypes.c_float(x["scale"]), P(g["do"]), P(g["dv_in"]), P(g["dht"]), P(dhck),
                            P(dv2), P(dh0), ctypes.byref(dims), P(ws), ws.numel(),
                            ctypes.c_void_p(stream.cuda_stream))
        if rc != 0:
            raise RuntimeError(kda.status_string(rc))

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if kda.status(ws, stream) != 0:
        raise RuntimeError("kernel status")
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.mark_start()
    per, span_ms = time_steps(step, args.steps, stream)
    clocks.mark_end()
    barrier(world)
    med = statistics.median(per)
    window_steps = clock_window(step, med, clocks)
    clk = clocks.stop()
    clk["clock_window_steps"] = window_steps
    ms_per_step = max_over_ranks(med, world)
    tokens = B * T if x["cu_seqlens"] is None else int(x["cu_seqlens"][-1])
    value = tokens * world / (ms_per_step / 1e3)
    hbm, _, _, peak_kind = peaks()
    th = tokens * H
    state = N * H * K * V * 4 * (2 if gr["dht"] is not None else 1)
    by = bwd_bytes_per_token_head(K, V) * th + state
    avg = med
    achieved = by / (avg / 1e3) / 1e9
    traffic = ncu_traffic("kda_bwd_dh_kernel", os.path.join(ROOT, "chunked_gated_delta_gb300", "csrc",
                                                            "bwd_dh.cu"), w.name)

    # end to end through the public API: upstream gradients from pinned host
    # memory, dv2 and dh0 back to pinned host memory (dhck stays on the device
    # for the next backward stage)
    e2e = None
    if args.e2e_steps > 0:
        hin = {n: (t.pin_memory() if t is not None else None) for n, t in gr.items()}
        dv2_h = torch.empty(dv2.shape, dtype=dv2.dtype, pin_memory=True)
        dh0_h = torch.empty(dh0.shape, dtype=dh0.dtype, pin_memory=True)
        h2d = sum(t.numel() * t.element_size() for t in hin.values() if t is not None)
        d2h = dv2_h.numel() * 2 + dh0_h.numel() * 4

        def one():
            for n, t in hin.items():
                if t is not None:
                    g[n].copy_(t, non_blocking=True)
            step()
            dv2_h.copy_(dv2, non_blocking=True)
            dh0_h.copy_(dh0, non_blocking=True)

        one()
        torch.cuda.synchronize(dev)
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        steps = max(1, min(args.steps, args.e2e_steps))
        e0.record(stream)
        for _ in range(steps):
            one()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = max_over_ranks(e0.elapsed_time(e1) / steps, world)
        e2e = {"value": tokens * world / (ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": steps,
               "path": "pinned host -> device (do, dv_in, dht), kda_bwd_dh, device -> pinned host (dv2, dh0)"}
    line = {
        "metric": BWD_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; forward workload inputs plus N(0,1) upstream gradients)",
        "config": {**workload_config(w, x), "path": "bwd_dh"},
        "timing": {"ms_per_step_median": ms_per_step, "ms_p10": pct(per, 0.1), "ms_p90": pct(per, 0.9),
                   "ms_per_step_mean": span_ms / args.steps, "per_step_events": True},
        "roofline": {"bound": "hbm", "kernel": "kda_bwd_dh_kernel", "achieved": achieved, "peak": hbm,
                     "unit": "GB/s", "frac": achieved / hbm, "traffic": traffic, "peak_kind": peak_kind,
                     "algorithmic_bytes_per_launch": by, "avg_launch_ms": avg},
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline:
        r, desc, _ = oracle_bwd_sample_rate(x, gr, args.ref_seconds)
        line["cpu_baseline"] = {"value": r, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": desc}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_e2e(args, kda, x, dims, stream, dev, world):
    """Same metric end to end through the host-buffer C-ABI call (kda_fwd_host):
    inputs in pinned host memory, outputs back to pinned host memory, all
    copies inside the timed region."""
    import torch
    names = ("q", "k", "v", "g", "beta")
    host_in = {n: x[n].pin_memory() for n in names}
    h0_host = x["h0"].pin_memory() if x["h0"] is not None else None
    cu_host = x["cu_seqlens"]
    B, T, H, K, V, N = x["B"], x["T"], x["H"], x["K"], x["V"], x["N"]
    o_host = torch.empty((B, T, H, V), dtype=torch.bfloat16, pin_memory=True)
    ht_host = torch.empty((N, H, K, V), dtype=torch.float32, pin_memory=True)
    arena = torch.empty(kda.host_arena_size(dims), dtype=torch.uint8, device=dev)
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    h2d += 0 if h0_host is None else h0_host.numel() * 4
    h2d += 0 if cu_host is None else cu_host.numel() * 4
    d2h = o_host.numel() * 2 + ht_host.numel() * 4
    steps = max(1, min(args.steps, args.e2e_steps))

    def one():
        kda.fwd_host(host_in["q"], host_in["k"], host_in["v"], host_in["g"], host_in["beta"], x["scale"],
                     h0_host, cu_host, o_host, ht_host, dims, arena, stream)

    one()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        one()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(e0.elapsed_time(e1) / steps, world)
    del arena
    return {"value": B * T * world / (ms / 1e3), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "steps": steps, "path": "kda_fwd_host: pinned host -> device copies, both kernels, "
                                    "device -> pinned host, one C-ABI call per step"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 200 on the GPU, long enough for in-region clock samples; "
                         "5 for the reference arm, whose steps are seconds of host work)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    ap.add_argument("--workload", default="headline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-seconds", type=float, default=2.0,
                    help="target wall seconds of one bounded oracle sample")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-configs", dest="configs", action="store_false",
                    help="skip the extra per-workload lines (mid, varlen, long) of the forward")
    ap.add_argument("--plan", choices=("auto", "fused"), default="auto",
                    help="auto: the two-stage forward (default); fused: the single-pass kernel "
                         "(KDA_PLAN_FUSED), timed against the strict single-pass I/O bound")
    ap.add_argument("--path", choices=("fwd", "bwd_dh"), default="fwd",
                    help="fwd: the forward (default); bwd_dh: the reverse state scan")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = 5 if args.impl == "reference" else 200
    if args.warmup < 3 and args.impl == "gb300":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        return run_reference(args)
    return run_gb300_bwd(args) if args.path == "bwd_dh" else run_gb300(args)


if __name__ == "__main__":
    sys.exit(main())
