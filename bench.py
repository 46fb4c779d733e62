#!/usr/bin/env python3
"""Throughput benchmark of the exact-attention library on GB300.

One step is one pass of the whole hot path over one batch of seeded synthetic
input: the forward kernel, and for the forward+backward workload the backward
call (row-dot preprocess, backward kernel, dQ postprocess).  The default
workload is B=2, H=16, N=4096, d=64, causal, forward + backward.

Prints ONE JSON line (rank 0).  ``value`` is algorithmic TFLOP/s of the whole
job (4 L^2 d per (sequence, head) forward, halved under the causal mask,
backward 2.5x that) with inputs resident in HBM; L2 is flushed before every
timed step (``flush_l2``).  ``e2e`` repeats the measurement through the same C
ABI with every step's inputs copied from pinned host memory and its gradients
(or O) copied back inside the timed region, the copies of neighbouring steps
overlapping the computation as in a training loop.  ``gpu_launches`` is the
library's own count of the kernels it launched inside the timed region.

``--impl reference`` times the fp64 CPU oracle (the only reference this method
has) on a bounded sample of the same workload.

``--workload decode_...`` measures one decoding step instead (one new query per
sequence against a resident K/V cache, split-K/V kernel plus combine): the
metric is algorithmic GB/s (K/V cache, q, o, LSE moved once) and the roofline
is HBM bandwidth.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "fwdbwd_b2_h16_n4096_d64_causal"
L2_NOTE = "flushed before every timed step (256 MiB write, then read back: no dirty line left)"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
THROTTLE_BITS = {  # nvidia-smi clocks_event_reasons bitmask
    0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
    0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
    0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting",
}


def flush_l2(buf, sink, value):
    """Evict L2 before a timed step, outside its events: write ``buf`` (256 MiB,
    twice the 129 MB L2), then read it back.  The write alone leaves L2 full of
    the flush's own dirty lines, and the timed step would then pay for writing
    them back to HBM (about 10 us of a 64 x 4096 decoding step); after the read
    L2 holds clean lines of the flush buffer and none of the step's data."""
    import torch

    buf.fill_(float(value))
    torch.sum(buf, dim=0, out=sink)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.t_on = self.t_off = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu),
                 "--query-gpu=timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), line.strip()))

    def mark_on(self):
        self.t_on = time.time()

    def mark_off(self):
        self.t_off = time.time()

    def stop_rows(self):
        if self.proc is not None:
            time.sleep(0.12)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return list(self.rows)

    def stop(self):
        return self.summarise(self.stop_rows(), self.t_on, self.t_off)

    @staticmethod
    def summarise(rows, t_on, t_off):
        sm, mx, reasons = [], [], set()
        for t, line in rows:
            if t_on is None or not (t_on - 0.06 <= t <= t_off + 0.06):
                continue
            parts = [p.strip() for p in line.split(",")]
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                bits = int(parts[4], 16)
            except (ValueError, IndexError):
                continue
            for b, name in THROTTLE_BITS.items():
                if bits & b:
                    reasons.add(name)
        reasons.discard("gpu_idle")
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def profile_entry(path, workload, kernel, key):
    """Field `key` of the committed ncu summary entry (profiles/traffic.json)
    for `kernel` on `workload`, or None."""
    if not path or not os.path.exists(path):
        return None
    with open(path) as f:
        entries = json.load(f).get("entries", [])
    for e in entries:
        if e.get("workload") == workload and e.get("kernel") == kernel:
            return e.get(key)
    return None


def traffic_entry(path, workload, kernel):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summary (profiles/traffic.json), or None."""
    return profile_entry(path, workload, kernel, "bytes_per_launch")


def step_stats(step_ms):
    """Median and 90th percentile of per-step event times (ms)."""
    xs = sorted(step_ms)
    return {"ms_median": round(statistics.median(xs), 4),
            "ms_p90": round(xs[min(len(xs) - 1, int(0.9 * len(xs)))], 4)}


def max_over_ranks(pg, values, device):
    """Each value's maximum over all ranks: the job takes as long as its
    slowest rank.  pg is torch.distributed (or None for one process)."""
    if pg is None:
        return [float(x) for x in values]
    import torch
    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return [float(x) for x in t]


def job_rate(units_per_step, steps, world, total_ms):
    """Whole-job throughput: every rank processes units_per_step per step
    (weak scaling: replicas, no data-path collective), over the slowest
    rank's time."""
    return units_per_step * steps * world / (total_ms * 1e-3)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def bench_ours(args, world, rank, local):
    import torch

    import exact_attention_21_gb300.fa as fa
    from exact_attention_21_gb300.inputs import WORKLOADS, make_inputs

    w = WORKLOADS[args.workload]
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    fa.lib()
    stream = torch.cuda.current_stream()

    host = make_inputs(w, seed=rank)  # weak scaling: each rank its own batch
    d, T, Hq, Hkv = w.d, w.T, w.Hq, w.Hkv
    cu = host["cu_seqlens"].to(dev) if w.varlen else None
    B, N = (len(w.seq_lengths), w.N) if w.varlen else (w.B, w.N)
    q, k, v = (host[n].to(dev) for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty(Hq, T, dtype=torch.float32, device=dev)
    if w.backward:
        do = host["do"].to(dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(fa.fa_bwd_workspace_size(Hq, T, d), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        fa.fa_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, T, w.scale, w.causal, cu, stream)
        if ev is not None:
            ev[1].record(stream)
        if w.backward:
            fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, B, Hq, Hkv, N, d, T, w.scale, w.causal, cu, ws, stream)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    fa.fa_stream_status(stream)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.15)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    sampler.mark_on()
    launches0 = fa.fa_launch_count()
    for i in range(args.steps):
        flush_l2(flush, sink, i)  # outside the timed events
        step(events[i])
    launches = fa.fa_launch_count() - launches0
    torch.cuda.synchronize()
    sampler.mark_off()
    if pg:
        pg.barrier()
    clocks = sampler.stop()
    fa.fa_stream_status(stream)
    fwd_ms = [e[0].elapsed_time(e[1]) for e in events]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in events]
    step_ms = [a + b for a, b in zip(fwd_ms, bwd_ms)]
    total_ms = sum(step_ms)

    # ---- end to end: every step's inputs copied in from pinned host memory and
    # its gradients (or O) copied back, through the same C ABI.  The steps are
    # pipelined as a training loop would run them: two device buffer sets, the
    # host-to-device copies of step i+1 and the device-to-host copies of step
    # i-1 on their own streams while step i computes.  The timed region spans
    # all copies of all steps.
    pin = {n: host[n].pin_memory() for n in host if n != "cu_seqlens"}
    outs = ("dq", "dk", "dv") if w.backward else ("o",)
    res_host = {n: torch.empty((T, Hq if n in ("dq", "o") else Hkv, d), dtype=torch.bfloat16).pin_memory()
                for n in outs}
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    d2h = sum(t.numel() * t.element_size() for t in res_host.values())
    e2e_steps = max(20, args.steps)
    sets = []
    for b in range(2):
        sset = {n: torch.empty_like(pin[n], device=dev) for n in pin}
        sset["o"] = torch.empty_like(sset["q"])
        sset["lse"] = torch.empty(Hq, T, dtype=torch.float32, device=dev)
        if w.backward:
            sset.update(dq=torch.empty_like(sset["q"]), dk=torch.empty_like(sset["k"]), dv=torch.empty_like(sset["v"]))
        sets.append(sset)
    h2d_stream, d2h_stream = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_steps_run(n):
        for i in range(n):
            b = i % 2
            S = sets[b]
            with torch.cuda.stream(h2d_stream):
                if i >= 2:
                    h2d_stream.wait_event(ev_done[b])  # step i-2's kernels have read these inputs
                for name, t in pin.items():
                    S[name].copy_(t, non_blocking=True)
                ev_in[b].record(h2d_stream)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])  # step i-2's results have been copied out of these outputs
            fa.fa_fwd(S["q"], S["k"], S["v"], S["o"], S["lse"], B, Hq, Hkv, N, d, T, w.scale, w.causal, cu, stream)
            if w.backward:
                fa.fa_bwd(S["q"], S["k"], S["v"], S["o"], S["do"], S["lse"], S["dq"], S["dk"], S["dv"], B, Hq, Hkv, N,
                          d, T, w.scale, w.causal, cu, ws, stream)
            ev_done[b].record(stream)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(ev_done[b])
                for name, t in res_host.items():
                    t.copy_(S[name], non_blocking=True)
                ev_out[b].record(d2h_stream)

    e2e_steps_run(2)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    e0.record(h2d_stream)
    e2e_steps_run(e2e_steps)
    e1.record(d2h_stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    fa.fa_stream_status(stream)

    total_ms, e2e_ms = max_over_ranks(pg, [total_ms, e2e_ms], dev)

    flops_step = w.fwd_flops() + (w.bwd_flops() if w.backward else 0.0)
    value = job_rate(flops_step, args.steps, world, total_ms) / 1e12
    e2e_value = job_rate(flops_step, 1, world, e2e_ms) / 1e12

    peaks, peak_src = load_peaks()
    fwd_avg = statistics.mean(fwd_ms)
    # q, k, v read and o written once (bf16), and the LSE (f32)
    fwd_bytes = 2 * T * d * (2 * Hq + 2 * Hkv) + 4 * Hq * T
    bwd_avg = statistics.mean(bwd_ms) if w.backward else 0.0
    if w.backward and bwd_avg > fwd_avg:
        kern, kflops, kms = "fa_bwd (row-dot, backward kernel, dQ convert)", w.bwd_flops(), bwd_avg
    else:
        kern, kflops, kms = "fa_fwd_kernel", w.fwd_flops(), fwd_avg
    achieved = kflops / (kms * 1e-3) / 1e12
    peak = peaks.get("bf16_tflops", PEAKS_FALLBACK["bf16_tflops"])
    line = {
        "metric": "attention fwd+bwd TFLOPS (bf16, 1xGB300) and % of dense BF16 tensor peak"
        if w.backward else "attention fwd TFLOPS (bf16, 1xGB300) and % of dense BF16 tensor peak",
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16)",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N, "d": d,
                   "causal": w.causal, "seq_lengths": w.seq_lengths if w.varlen else None,
                   "global_batch": w.B * world, "seq_len": w.N,
                   "fwd_gflop_per_step": round(w.fwd_flops() / 1e9, 3),
                   "bwd_gflop_per_step": round(w.bwd_flops() / 1e9, 3) if w.backward else 0.0,
                   "l2": L2_NOTE,
                   "parallelism": f"replicas x{world}"},
        "fwd_ms": round(fwd_avg, 4),
        "bwd_ms": round(bwd_avg, 4),
        "pct_of_bf16_peak": round(100 * value / world / peak, 2),
        "roofline": {"bound": "tensor", "kernel": kern, "achieved": round(achieved, 2), "peak": peak,
                     "peak_source": f"{peak_src} bf16_tflops (burst)", "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": None,
                     "frac_of_sustained": round(achieved / peaks.get("bf16_tflops_sustained",
                                                                      PEAKS_FALLBACK["bf16_tflops_sustained"]), 4)},
        "step_times": step_stats(step_ms),
        "algorithmic_gbs_fwd": round(fwd_bytes / (fwd_avg * 1e-3) / 1e9, 1),
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "pipelining": "two buffer sets; copies in and out on their own streams overlap the neighbouring steps"},
        "gpu_launches": launches,
        "clocks": clocks,
    }
    tr = traffic_entry(args.traffic_file, w.name, kern)
    if tr is not None:
        line["roofline"]["traffic"] = tr
    pt = profile_entry(args.traffic_file, w.name, kern, "pipe_tensor_pct")
    if pt is not None:
        line["roofline"]["pipe_tensor_pct"] = pt
    if not args.no_per_config and w.name == DEFAULT_WORKLOAD:
        del sets, pin, res_host, q, k, v, o, lse, host
        if w.backward:
            del do, dq, dk, dv, ws
        torch.cuda.empty_cache()
        line["per_config"] = per_config_lines(args, rank, dev, stream, flush, sink, peaks)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_seconds)
    if pg:
        pg.destroy_process_group()
    return line if rank == 0 else None


# The other workloads of the headline table, measured in the default run with
# the pages' protocol: 20 warm-ups, then timed runs (at least 50, and enough
# for a few clock samples), L2 flushed before each, median and P90.
PER_CONFIG = ("fwd_b1_h1_n256_d64", "fwd_b4_h16_n2048_d64", "fwd_b2_h32_n4096_d128_causal",
              "fwd_varlen8_hq32_hkv8_d128_causal", "decode_b64_hq64_hkv8_n4096_d128",
              "decode_b64_hq64_hkv8_n4096_d64", "decode_varlen8_hq32_hkv8_d128")


def per_config_lines(args, rank, dev, stream, flush, sink, peaks):
    import torch

    import exact_attention_21_gb300.fa as fa
    from exact_attention_21_gb300.inputs import WORKLOADS, make_inputs

    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.15)
    out = {}
    for name in PER_CONFIG:
        w = WORKLOADS[name]
        host = make_inputs(w, seed=rank, with_do=False)
        d, T, Hq, Hkv = w.d, w.T, w.Hq, w.Hkv
        cu = host["cu_seqlens"].to(dev) if w.varlen else None
        B, N = (len(w.seq_lengths), w.N) if w.varlen else (w.B, w.N)
        q, k, v = (host[n].to(dev) for n in ("q", "k", "v"))
        del host
        o = torch.empty_like(q)
        if w.decode:
            lse = torch.empty(Hq, B, dtype=torch.float32, device=dev)
            ws = torch.empty(fa.fa_decode_workspace_size(B, Hq, d, N), dtype=torch.uint8, device=dev)

            def run():
                fa.fa_decode(q, k, v, o, lse, B, Hq, Hkv, N, d, T, w.scale, cu, ws, stream)
        else:
            lse = torch.empty(Hq, T, dtype=torch.float32, device=dev)

            def run():
                fa.fa_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, T, w.scale, w.causal, cu, stream)
        for _ in range(20):
            run()
        fa.fa_stream_status(stream)
        # size the timed loop: at least 50 runs and about 0.3 s under load
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(5):
            flush_l2(flush, sink, 1.0)
            run()
        e1.record(stream)
        torch.cuda.synchronize()
        per_iter_s = e0.elapsed_time(e1) * 1e-3 / 5
        n = int(min(5000, max(50, 0.3 / max(per_iter_s, 1e-6))))
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        torch.cuda.synchronize()
        t_on = time.time()
        for i in range(n):
            flush_l2(flush, sink, i)
            evs[i][0].record(stream)
            run()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        t_off = time.time()
        fa.fa_stream_status(stream)
        ms = sorted(a.elapsed_time(b) for a, b in evs)
        med, p90 = statistics.median(ms), ms[min(n - 1, int(0.9 * n))]
        entry = {"runs": n, "us_median": round(med * 1e3, 2), "us_p90": round(p90 * 1e3, 2)}
        if w.decode:
            nbytes = w.decode_bytes()
            gbs = nbytes / (med * 1e-3) / 1e9
            entry.update(kernel="fa_decode (split kernel + combine)", bytes=nbytes, gbs=round(gbs, 1),
                         frac_of_hbm=round(gbs / peaks.get("hbm_gbs", PEAKS_FALLBACK["hbm_gbs"]), 4))
        else:
            flops = w.fwd_flops()
            nbytes = 2 * T * d * (2 * Hq + 2 * Hkv) + 4 * Hq * T
            tf = flops / (med * 1e-3) / 1e12
            entry.update(kernel="fa_fwd_kernel", gflop=round(flops / 1e9, 3), tflops=round(tf, 1),
                         frac=round(tf / peaks.get("bf16_tflops", PEAKS_FALLBACK["bf16_tflops"]), 4),
                         frac_of_sustained=round(
                             tf / peaks.get("bf16_tflops_sustained", PEAKS_FALLBACK["bf16_tflops_sustained"]), 4),
                         bytes=nbytes, gbs=round(nbytes / (med * 1e-3) / 1e9, 1))
        pt = profile_entry(args.traffic_file, name, entry["kernel"], "pipe_tensor_pct")
        if pt is not None:
            entry["pipe_tensor_pct"] = pt
        entry["window"] = (t_on, t_off)
        out[name] = entry
        del q, k, v, o, lse
        if w.decode:
            del ws
        torch.cuda.empty_cache()
    rows = sampler.stop_rows()
    for entry in out.values():
        t_on, t_off = entry.pop("window")
        entry["clocks"] = ClockSampler.summarise(rows, t_on, t_off)
    return out


DECODE_METRIC = "attention decode step, K/V cache bytes read per second (1xGB300)"


def bench_decode(args, world, rank, local):
    """One decoding step per timed iteration: fa_decode (split kernel +
    combine) over a K/V cache resident in HBM, larger than L2 for the
    64-sequence workload; L2 is flushed before every step anyway."""
    import torch

    import exact_attention_21_gb300.fa as fa
    from exact_attention_21_gb300.inputs import WORKLOADS, make_inputs

    w = WORKLOADS[args.workload]
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    fa.lib()
    stream = torch.cuda.current_stream()
    host = make_inputs(w, seed=rank)
    d, T, Hq, Hkv, B, N = w.d, w.T, w.Hq, w.Hkv, w.B, w.N
    cu = host["cu_seqlens"].to(dev) if w.varlen else None
    q, k, v = (host[n].to(dev) for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty(Hq, B, dtype=torch.float32, device=dev)
    ws = torch.empty(fa.fa_decode_workspace_size(B, Hq, d, N), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)
    if w.page_size:
        # the cache lives in pages scattered over a pool, reached through the table
        k, v = host["k_pages"].to(dev), host["v_pages"].to(dev)
        table, seqlens = host["block_table"].to(dev), host["seqlens"].to(dev)
    if w.fp8:
        # the cache is quantised when it is written, before the decoding steps
        k8, ks = fa.kv_quantize_fp8(k)
        v8, vs = fa.kv_quantize_fp8(v)
        del k, v

    def step():
        if w.page_size and w.fp8:
            fa.fa_decode_paged_fp8(q, k8, v8, ks, vs, table, seqlens, o, lse, w.page_size, w.scale, ws, stream)
        elif w.page_size:
            fa.fa_decode_paged(q, k, v, table, seqlens, o, lse, w.page_size, w.scale, ws, stream)
        elif w.fp8:
            fa.fa_decode_fp8(q, k8, v8, ks, vs, o, lse, B, Hq, Hkv, N, d, T, w.scale, cu, ws, stream)
        else:
            fa.fa_decode(q, k, v, o, lse, B, Hq, Hkv, N, d, T, w.scale, cu, ws, stream)

    for _ in range(args.warmup):
        step()
    fa.fa_stream_status(stream)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.15)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    sampler.mark_on()
    launches0 = fa.fa_launch_count()
    for i in range(args.steps):
        flush_l2(flush, sink, i)
        events[i][0].record(stream)
        step()
        events[i][1].record(stream)
    launches = fa.fa_launch_count() - launches0
    torch.cuda.synchronize()
    sampler.mark_off()
    if pg:
        pg.barrier()
    clocks = sampler.stop()
    fa.fa_stream_status(stream)
    step_ms = [e[0].elapsed_time(e[1]) for e in events]
    total_ms = sum(step_ms)

    # end to end: the step's query from pinned host memory in, O and the LSE
    # back; the K/V cache stays resident, as it does between decoding steps
    q_pin = host["q"].pin_memory()
    o_host = torch.empty_like(host["q"]).pin_memory()
    l_host = torch.empty(Hq, B, dtype=torch.float32).pin_memory()
    h2d = q_pin.numel() * q_pin.element_size()
    d2h = o_host.numel() * o_host.element_size() + l_host.numel() * 4
    e2e_steps = max(20, args.steps)

    def e2e_step():
        q.copy_(q_pin, non_blocking=True)
        step()
        o_host.copy_(o, non_blocking=True)
        l_host.copy_(lse, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    # each step is timed from the copy of its query in to the copies of its
    # results out, with L2 flushed before it outside the events, as for ``value``
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(e2e_steps)]
    for i in range(e2e_steps):
        flush_l2(flush, sink, i)
        e2e_ev[i][0].record(stream)
        e2e_step()
        e2e_ev[i][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = sum(a.elapsed_time(b) for a, b in e2e_ev) / e2e_steps
    fa.fa_stream_status(stream)
    total_ms, e2e_ms = max_over_ranks(pg, [total_ms, e2e_ms], dev)

    nbytes = w.decode_bytes()
    value = job_rate(nbytes, args.steps, world, total_ms) / 1e9
    avg_ms = total_ms / args.steps
    peaks, peak_src = load_peaks()
    peak = peaks.get("hbm_gbs", PEAKS_FALLBACK["hbm_gbs"])
    achieved = nbytes / (avg_ms * 1e-3) / 1e9
    line = {
        "metric": DECODE_METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(avg_ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 cache, f16 products" if w.fp8 else "bf16",
        "data": "synthetic (seeded N(0,1) bf16)",
        "config": {"workload": w.name, "B": B, "Hq": Hq, "Hkv": Hkv, "N": N, "d": d,
                   "seq_lengths": w.seq_lengths if w.varlen else None, "queries_per_sequence": 1,
                   "kv_cache": ("E4M3 codes + f32 per-token scales" if w.fp8 else "bf16")
                   + (f", pages of {w.page_size} tokens at random pool positions" if w.page_size else ""),
                   "kv_cache_bytes": w.kv_cache_bytes(), "bytes_per_step": nbytes,
                   "gflop_per_step": round(w.decode_flops() / 1e9, 3),
                   "tokens_per_s": round(B * world / (avg_ms * 1e-3), 1),
                   "l2": L2_NOTE,
                   "parallelism": f"replicas x{world}"},
        "step_times": step_stats(step_ms),
        "roofline": {"bound": "hbm", "kernel": "fa_decode" + ("_paged" if w.page_size else "") + ("_fp8" if w.fp8 else "")
                     + " (split kernel + combine)",
                     "achieved": round(achieved, 1),
                     "peak": peak, "peak_source": f"{peak_src} hbm_gbs", "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": None},
        "e2e": {"value": round(job_rate(nbytes, 1, world, e2e_ms) / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": launches,
        "clocks": clocks,
    }
    tr = traffic_entry(args.traffic_file, w.name, line["roofline"]["kernel"])
    if tr is not None:
        line["roofline"]["traffic"] = tr
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_decode(w, budget_s=args.cpu_seconds)
    if pg:
        pg.destroy_process_group()
    return line if rank == 0 else None


def oracle_decode_sample(w, n_seq, seed=0):
    """fp64 oracle on the first n_seq sequences of decoding workload w (every
    head); returns (seconds, algorithmic bytes of that sample)."""
    import numpy as np
    import torch

    import oracle
    from exact_attention_21_gb300.inputs import make_decode_qkv

    lens = w.seq_lengths[:n_seq]
    T = int(sum(lens))
    t = make_decode_qkv(n_seq, w.Hq, T, w.Hkv, w.d, seed=seed)
    f64 = {n: t[n].to(torch.float64).numpy() for n in t}
    cu = oracle.cu_from_lengths(lens)
    if w.fp8:
        from oracle import quant
        k8, ks = quant.quantize_rows_fp8(t["k"].float().numpy())
        v8, vs = quant.quantize_rows_fp8(t["v"].float().numpy())
    t0 = time.perf_counter()
    if w.fp8:
        oracle.attention_decode(f64["q"], quant.dequantize_rows_fp8(k8, ks), quant.dequantize_rows_fp8(v8, vs), cu,
                                w.scale)
    else:
        oracle.attention_decode(f64["q"], f64["k"], f64["v"], cu, w.scale)
    sec = time.perf_counter() - t0
    per_tok = 2 * w.Hkv * ((w.d + 4) if w.fp8 else 2 * w.d)
    nbytes = T * per_tok + 2 * n_seq * w.Hq * w.d * 2 + n_seq * w.Hq * 4
    return sec, nbytes


def cpu_baseline_decode(w, budget_s=15.0):
    sec1, b1 = oracle_decode_sample(w, 1)
    n = max(1, min(w.B, int(budget_s / max(sec1, 1e-3))))
    sec, nb = oracle_decode_sample(w, n) if n > 1 else (sec1, b1)
    return {"value": round(nb / sec / 1e9, 4), "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{n} of {w.B} sequences of {w.name} (every head), numpy fp64 (BLAS threads = all host cores)",
            "seconds": round(sec, 3)}


def oracle_sample(w, n_heads, seed=0):
    """Runs the fp64 oracle on the first n_heads (sequence, query head) pairs of
    workload w; returns (seconds, algorithmic flops of that sample)."""
    import numpy as np
    import torch

    import oracle
    from exact_attention_21_gb300.inputs import make_qkv

    L = w.seq_lengths[0]
    t = make_qkv(L, n_heads, n_heads, w.d, seed=seed, with_do=w.backward)
    f64 = {n: t[n].to(torch.float64).numpy() for n in t}
    cu = np.array([0, L])
    t0 = time.perf_counter()
    oracle.attention_forward(f64["q"], f64["k"], f64["v"], cu, w.scale, w.causal)
    if w.backward:
        oracle.attention_backward(f64["q"], f64["k"], f64["v"], f64["do"], cu, w.scale, w.causal)
    sec = time.perf_counter() - t0
    per_head = 4.0 * L * L * w.d / (2 if w.causal else 1)
    flops = per_head * n_heads * (3.5 if w.backward else 1.0)
    return sec, flops


def cpu_baseline(w, budget_s=15.0):
    sec1, fl1 = oracle_sample(w, 1)
    n = max(1, min(w.Hq, int(budget_s / max(sec1, 1e-3))))
    sec, fl = oracle_sample(w, n) if n > 1 else (sec1, fl1)
    return {"value": round(fl / sec / 1e12, 6), "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{n} of {w.Hq * len(w.seq_lengths)} (sequence, head) pairs of {w.name}, L={w.seq_lengths[0]}, "
                      f"numpy fp64 (BLAS threads = all host cores)",
            "seconds": round(sec, 3)}


def bench_reference(args, world, rank):
    from exact_attention_21_gb300.inputs import WORKLOADS

    if rank != 0:
        return None
    w = WORKLOADS[args.workload]
    if w.decode:
        for _ in range(args.warmup):
            oracle_decode_sample(w, 1)
        secs, nbytes = 0.0, 0
        for _ in range(args.steps):
            s_, b_ = oracle_decode_sample(w, 1)
            secs += s_
            nbytes += b_
        value = nbytes / secs / 1e9
        sample = f"1 sequence (every head) of {w.name} per step, numpy fp64 (BLAS threads = all host cores)"
        return {
            "impl": "reference", "metric": DECODE_METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * secs / args.steps, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1) bf16)",
            "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N, "d": w.d,
                       "parallelism": "cpu oracle, rank 0 only"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
    for _ in range(args.warmup):
        oracle_sample(w, 1)
    secs, flops = 0.0, 0.0
    for _ in range(args.steps):
        s, f = oracle_sample(w, 1)
        secs += s
        flops += f
    value = flops / secs / 1e12
    sample = f"1 (sequence, head) pair of {w.name} per step, numpy fp64 (BLAS threads = all host cores)"
    return {
        "impl": "reference",
        "metric": "attention fwd+bwd TFLOPS (bf16, 1xGB300) and % of dense BF16 tensor peak"
        if w.backward else "attention fwd TFLOPS (bf16, 1xGB300) and % of dense BF16 tensor peak",
        "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * secs / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1) bf16)",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N, "d": w.d,
                   "causal": w.causal, "parallelism": "cpu oracle, rank 0 only"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-config forward / decode lines of the default run")
    ap.add_argument("--traffic-file", default=os.path.join(ROOT, "profiles", "traffic.json"))
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    from exact_attention_21_gb300.inputs import WORKLOADS
    if args.workload not in WORKLOADS:
        ap.error(f"unknown workload {args.workload}; one of {sorted(WORKLOADS)}")
    if args.impl == "reference":
        line = bench_reference(args, world, rank)
    elif WORKLOADS[args.workload].decode:
        line = bench_decode(args, world, rank, local)
    else:
        line = bench_ours(args, world, rank, local)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
