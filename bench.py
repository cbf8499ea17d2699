#!/usr/bin/env python3
"""Benchmark of the Transformer-XL relative-attention hot path on GB300.

One step = one pass of the whole hot path over one batch: for every segment
and every layer of the workload, the fused relative-attention kernel
(txl_attn_fwd) followed by the in-place Tail_M memory roll (txl_mem_update),
in the multi-segment driver's order, on one stream.  The per-call inputs
(Q, K, V projected by the harness, the layer input h) are produced once by
running the chain (projections in fp32 on the GPU with TF32 off, cast to
bf16) and stay resident in HBM; a step replays the launch sequence over
them as one CUDA graph.  Each step reads more than the 129 MB L2 holds
(several GB for the default workload), so no explicit flush is needed.

Output: one JSON line on rank 0 (see the keys below).  ``--impl reference``
times the fp64 CPU oracle instead (the reference arm of this method).

Multi-GPU: the path shards over independent replicas (batch rows carry their
own memories; there is no exchange step), so N ranks each run the same
workload (weak scaling) and ``value`` = units of all ranks / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import shutil
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import txl_workloads as W  # noqa: E402

METRIC = "rel-attn TFLOP/s & tokens/s per segment (1×GB300) and % of bf16 tensor peak"
DEFAULT_WORKLOAD = "base512_bf16"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# --------------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(elapsed_ms_local: float, ws: int, work_per_step: float, steps: int):
    """Whole-job throughput over ``ws`` replicas that each did ``work_per_step``
    per step: the slowest rank's time (max over ranks) divides the work of all
    ranks.  Returns (rate per second, max elapsed ms)."""
    elapsed_max = reduce_max(elapsed_ms_local, ws)
    return ws * work_per_step * steps / (elapsed_max * 1e-3), elapsed_max


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


class ClockSampler:
    """Samples SM clock, power and throttle reasons with nvidia-smi while the
    timed region runs."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        self.t_start = self.t_stop = None
        exe = shutil.which("nvidia-smi")
        if exe is None:
            return
        ident = None
        try:
            ident = str(torch.cuda.get_device_properties(device_index).uuid)
            if not ident.startswith("GPU-"):
                ident = "GPU-" + ident
        except Exception:
            ident = None
        cmd = [exe, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if ident:
            cmd += ["-i", ident]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except Exception:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append((time.time(), ln.strip()))

    def mark_start(self):
        self.t_start = time.time()

    def mark_stop(self):
        self.t_stop = time.time()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        rows = []
        for t, ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((t, float(parts[1]), float(parts[2]), parts[3], parts[4:9]))
            except ValueError:
                continue
        in_win = [r for r in rows if self.t_start and self.t_stop and
                  self.t_start - 0.05 <= r[0] <= self.t_stop + 0.05]
        use = in_win if in_win else rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in use:
            flags = r[4][1:]
            for nm, fl in zip(names, flags):
                if fl.lower() in ("active", "1"):
                    reasons.add(nm)
        pw = []
        for r in use:
            try:
                pw.append(float(r[3]))
            except ValueError:
                pass
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": sorted(reasons), "samples": len(use),
                "samples_in_timed_region": len(in_win),
                "power_w_max": max(pw) if pw else None}


# --------------------------------------------------------------------- our arm
def build_calls(wl: W.Workload, dev):
    """Runs the chain once (harness projections + our kernels) and returns the
    per-call resident inputs.  Layer n+1's input is the head-merged output of
    layer n; memories roll by Tail_M between segments."""
    import transformer_xl_relative_attn_gb300 as txl
    dt = wl.torch_dtype
    params = W.make_params(wl)
    lws = [W.LayerWeights(*(getattr(lw, f).to(dev) for f in ("W_q", "W_k", "W_v", "W_r")))
           for lw in params.layers]
    mems = [m.to(device=dev, dtype=dt) for m in W.initial_memories(wl)]
    mems0 = [m.clone() for m in mems]
    rks = [W.project_r(lw, wl.M, wl.L, wl.H, device=dev).to(dt) for lw in lws]
    u = params.u.to(device=dev, dtype=dt)
    vb = params.v.to(device=dev, dtype=dt)
    calls = []
    for s in range(wl.segments):
        h = W.segment_input(wl, s).to(device=dev, dtype=dt)
        for n in range(wl.layers):
            q, k, v = W.project_qkv(lws[n], mems[n], h, wl.H)
            q, k, v = q.to(dt), k.to(dt), v.to(dt)
            out = torch.empty_like(q)
            txl.attn_fwd(q, k, v, rks[n], u, vb, wl.scale, out=out)
            txl.mem_update(mems[n], h)
            calls.append({"n": n, "q": q, "k": k, "v": v, "h": h, "out": out})
            h = W.merge_heads(out)
    torch.cuda.synchronize()
    txl.check_status()
    for m, m0 in zip(mems, mems0):
        m.copy_(m0)
    return calls, mems, rks, u, vb


def run_ours(args, wl: W.Workload):
    import transformer_xl_relative_attn_gb300 as txl

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    txl.load()
    peaks, peak_src = load_peaks()

    calls, mems, rks, u, vb = build_calls(wl, dev)
    n_calls = len(calls)
    stream = torch.cuda.Stream(device=dev)

    ev_a = [torch.cuda.Event(enable_timing=True, external=True) for _ in calls]
    ev_b = [torch.cuda.Event(enable_timing=True, external=True) for _ in calls]

    side = torch.cuda.Stream(device=dev)
    # scratch of the split-key path (allocated once, outside the timed region;
    # none when the workload has enough items to fill the GPU)
    scratch_bytes = txl.attn_workspace_bytes(wl.B, wl.H, wl.L, wl.M, wl.dh)
    scratch = torch.empty(scratch_bytes, dtype=torch.uint8, device=dev) if scratch_bytes else None

    def step(timed_events: bool):
        # Attention calls in order on the current stream; each Tail_M roll on a
        # side stream, after the point where its layer's inputs were projected
        # (just before that layer's attention) and before the next segment's
        # layer of the same memory starts (the projection reads the rolled
        # memory).  The rolls (HBM-bound) thus overlap later attention calls
        # (tensor/ALU-bound), with every data dependency of the segment
        # recurrence kept.
        cur = torch.cuda.current_stream()
        rolled = {}
        for c, ea, eb in zip(calls, ev_a, ev_b):
            n = c["n"]
            if n in rolled:
                cur.wait_event(rolled[n])
            inputs_ready = torch.cuda.Event()
            inputs_ready.record(cur)
            if timed_events:
                ea.record()
            if scratch is None:
                txl.attn_fwd(c["q"], c["k"], c["v"], rks[n], u, vb, wl.scale, out=c["out"])
            else:
                txl.attn_fwd_ws(c["q"], c["k"], c["v"], rks[n], u, vb, scratch, wl.scale,
                                out=c["out"])
            if timed_events:
                eb.record()
            side.wait_event(inputs_ready)
            with torch.cuda.stream(side):
                txl.mem_update(mems[n], c["h"], stream=side)
            rolled[n] = torch.cuda.Event()
            rolled[n].record(side)
        joined = torch.cuda.Event()
        joined.record(side)
        cur.wait_event(joined)

    # capture one step as a CUDA graph (warm the launch path first)
    with torch.cuda.stream(stream):
        step(False)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step(True)
    torch.cuda.synchronize()

    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    txl.check_status()

    sampler = ClockSampler(dev.index)
    time.sleep(0.2)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    sampler.mark_start()
    t0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            graph.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    sampler.mark_stop()
    barrier(ws)
    time.sleep(0.1)
    sampler.stop()
    elapsed_ms = t0.elapsed_time(t1)
    attn_ms = [a.elapsed_time(b) for a, b in zip(ev_a, ev_b)]  # last replay of the timed region
    roll_avg_ms = time_rolls(calls, mems, stream)
    roll_long = time_longmem_rolls(dev, stream, peaks)
    proj = time_projections(wl, dev, stream, peaks)
    bwd = (time_backward(wl, calls, rks, u, vb, dev, float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])),
                         peak_src) if wl.dh <= 256 else None)
    txl.check_status()
    flops_call = wl.attn_flops()
    flops_step = flops_call * n_calls
    tokens_step = wl.B * wl.L * wl.segments
    rate, elapsed_max = whole_job_rate(elapsed_ms, ws, flops_step, args.steps)
    value = rate / 1e12
    ms_per_step = elapsed_max / args.steps
    attn_avg_ms = sum(attn_ms) / len(attn_ms)
    achieved = flops_call / (attn_avg_ms * 1e-3) / 1e12
    # the timed region is tens of milliseconds at the maximum SM clock (the
    # clock record below shows it): burst conditions, so the burst peak
    peak_tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))

    result = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if wl.dtype == "bf16" else "f32",
        "data": "synthetic (seeded N(0,1) hidden states and memories, N(0,0.02) weights, "
                "sinusoid R; harness projections)",
        "config": {
            "workload": wl.name, "B": wl.B, "H": wl.H, "d_h": wl.dh, "L": wl.L, "M": wl.M,
            "layers": wl.layers, "segments": wl.segments,
            "calls_per_step": {"txl_attn_fwd": n_calls, "txl_mem_update": n_calls},
            "global_batch": wl.B * ws, "seq_len": wl.L, "mem_len": wl.M,
            "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
            "l2": "inputs larger than L2: each step reads "
                  f"{sum(sum(c[x].numel() * c[x].element_size() for x in ('q', 'k', 'v', 'h')) for c in calls) / 1e9:.2f} GB",
            "step": "CUDA graph of all (segment, layer) attention + Tail_M launches",
        },
        "tokens_per_s": round(ws * tokens_step * args.steps / (elapsed_max * 1e-3), 1),
        "pct_bf16_peak": round(100.0 * value / ws / peak_tf, 2),
        "roofline": {
            "kernel": "attn_tc_bf16_kernel",
            "bound": "tensor",
            "achieved": round(achieved, 2),
            "peak": peak_tf,
            "unit": "TFLOP/s",
            "frac": round(achieved / peak_tf, 4),
            "traffic": measured_traffic(wl.name),
            "peak_source": f"bf16_tflops, burst ({peak_src}): the timed region is tens of ms at max clock",
            "flops_per_launch": flops_call,
            "avg_launch_ms": round(attn_avg_ms, 5),
            "launches_averaged": len(attn_ms),
            "attn_share_of_step": round(sum(attn_ms) / ms_per_step, 4),
        },
        # per call: the attention kernel (+ the split combine pass) and Tail_M
        # the Tail_M roll timed alone after the timed region (in the step it
        # runs on a second stream in the gaps between attention kernels)
        "projections": proj,
        "backward": bwd,
        "roofline_mem_update": {
            "kernel": "tail_copy_kernel" if wl.L >= wl.M else "tail_chain_kernel",
            "workload": wl.name,
            "bound": "hbm",
            "achieved": round(wl.mem_update_bytes() / (roll_avg_ms * 1e-3) / 1e9, 1),
            "peak": float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])),
            "unit": "GB/s",
            "frac": round(wl.mem_update_bytes() / (roll_avg_ms * 1e-3) / 1e9
                          / float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])), 4),
            "bytes_per_launch": wl.mem_update_bytes(),
            "avg_launch_ms": round(roll_avg_ms, 5),
            "measured": f"the step's {n_calls} rolls in step order, back to back in one CUDA graph, "
                        "events around the graph only (total / rolls, median of 5 replays)",
        },
        "roofline_mem_update_longmem3200": roll_long,
        "gpu_launches": (3 if scratch is not None else 2) * n_calls * args.steps,
        "clocks": sampler.summary(),
    }

    if not args.no_e2e:
        if wl.dh == 64 and wl.dtype == "bf16" and wl.H % 4 == 0 and wl.L % 128 == 0 and wl.M % 128 == 0:
            result["e2e"] = measure_e2e_stack(args, wl, dev, flops_step, ws)
            # the attention calls alone through the host: q, k, v, h of every
            # call copied in, every output copied out
            result["e2e_attn_calls"] = measure_e2e(args, wl, calls, stream, side, mems, rks, u, vb,
                                                   scratch, flops_step, ws)
            if wl.d % 256 == 0 and wl.d <= 2048:
                result["decoder_stack"] = measure_decoder(args, wl, dev, flops_step, ws)
        else:
            result["e2e"] = measure_e2e(args, wl, calls, stream, side, mems, rks, u, vb, scratch,
                                        flops_step, ws)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"], result["parity"] = cpu_baseline_and_parity(wl, calls, rks, u, vb)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one attention
# launch, from an ncu capture summarised under profiles/; reported only while
# the kernel sources still hash to what was captured.
_TRAFFIC_CAPTURES = {
    "base512_bf16": {
        "sha256_prefix": {"attn_tc_bf16.cu": "7dd2381a9b741c12", "txl_device.cuh": "77bcc7df07e42fb8",
                          "attn_tc_common.cuh": "a91b70485c74670f"},
        "bytes_per_launch": 60071552,
        "summary": "profiles/attn_tc_bf16_base512_ncu_full.md",
    },
}


def measured_traffic(workload):
    import hashlib

    cap = _TRAFFIC_CAPTURES.get(workload)
    if cap is None:
        return None
    csrc = os.path.join(ROOT, "transformer_xl_relative_attn_gb300", "csrc")
    for name, prefix in cap["sha256_prefix"].items():
        with open(os.path.join(csrc, name), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest()[:16] != prefix:
                return None
    return cap["bytes_per_launch"]


def time_projections(wl, dev, stream, peaks):
    """The layer projections that produce the attention's inputs (txl_qkv_proj:
    q from h, k/v from memory and h; txl_r_proj; and both in one launch,
    txl_qkvr_proj), timed alone for one layer of
    the workload in a captured graph (kernel time, not the host launch path).
    They are not part of the timed step: the step starts from projected
    inputs.  None when the sizes are outside the projection kernel's range."""
    import transformer_xl_relative_attn_gb300 as txl

    B, L, M, H, dh = wl.B, wl.L, wl.M, wl.H, wl.dh
    d = H * dh
    if dh != 64 or H % 4 or L % 128 or M % 128 or wl.dtype != "bf16":
        return None
    g = torch.Generator(device="cpu").manual_seed(17)
    h = torch.randn(B, L, d, generator=g).to(device=dev, dtype=torch.bfloat16)
    mem = torch.randn(B, M, d, generator=g).to(device=dev, dtype=torch.bfloat16)
    w = (0.02 * torch.randn(3 * d, d, generator=g)).to(device=dev, dtype=torch.bfloat16)
    emb = torch.randn(M + L, d, generator=g).to(device=dev, dtype=torch.bfloat16)
    wr = (0.02 * torch.randn(d, d, generator=g)).to(device=dev, dtype=torch.bfloat16)
    q = torch.empty(B, H, L, dh, dtype=torch.bfloat16, device=dev)
    k = torch.empty(B, H, M + L, dh, dtype=torch.bfloat16, device=dev)
    v = torch.empty_like(k)
    r = torch.empty(M + L, H, dh, dtype=torch.bfloat16, device=dev)
    reps = 10
    ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]
    with torch.cuda.stream(stream):
        txl.qkv_proj(h, mem, w, H, q, k, v)
        txl.r_proj(emb, wr, H, r)
        txl.qkvr_proj(h, mem, w, emb, wr, H, q, k, v, r)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        ev[0].record()
        for _ in range(reps):
            txl.qkv_proj(h, mem, w, H, q, k, v)
        ev[1].record()
        for _ in range(reps):
            txl.r_proj(emb, wr, H, r)
        ev[2].record()
        for _ in range(reps):
            txl.qkvr_proj(h, mem, w, emb, wr, H, q, k, v, r)
        ev[3].record()
    graph.replay()
    torch.cuda.synchronize()
    txl.check_status()
    qkv_ms = ev[0].elapsed_time(ev[1]) / reps
    r_ms = ev[1].elapsed_time(ev[2]) / reps
    qkvr_ms = ev[2].elapsed_time(ev[3]) / reps
    f_qkv = 2.0 * B * L * d * d + 2.0 * B * (M + L) * 2 * d * d
    f_r = 2.0 * (M + L) * d * d
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    return {
        "qkv_proj": {"ms": round(qkv_ms, 5), "tflops": round(f_qkv / (qkv_ms * 1e-3) / 1e12, 2),
                     "frac": round(f_qkv / (qkv_ms * 1e-3) / 1e12 / peak, 4), "flops": f_qkv},
        "r_proj": {"ms": round(r_ms, 5), "tflops": round(f_r / (r_ms * 1e-3) / 1e12, 2),
                   "frac": round(f_r / (r_ms * 1e-3) / 1e12 / peak, 4), "flops": f_r,
                   "note": "alone: a few tiles on 152 SMs (launch-bound)"},
        "qkvr_proj": {"ms": round(qkvr_ms, 5), "tflops": round((f_qkv + f_r) / (qkvr_ms * 1e-3) / 1e12, 2),
                      "frac": round((f_qkv + f_r) / (qkvr_ms * 1e-3) / 1e12 / peak, 4), "flops": f_qkv + f_r,
                      "note": "q, k|v and r of one layer in one launch (txl_qkvr_proj)"},
        "peak": peak, "peak_source": "bf16_tflops (burst: kernels timed alone)",
        "measured": "one layer's projections, 10 back-to-back repeats in a CUDA graph",
    }


def time_rolls(calls, mems, stream, reps=5):
    """Average duration (ms) of one Tail_M roll: every call's roll of the step,
    in step order (consecutive rolls touch different layers' memories and
    different hidden states), back to back on `stream` as one CUDA graph with
    CUDA events only around the whole sequence; the graph is replayed
    ``reps`` times and the median replay is divided by the number of rolls."""
    import transformer_xl_relative_attn_gb300 as txl

    t0 = torch.cuda.Event(enable_timing=True, external=True)
    t1 = torch.cuda.Event(enable_timing=True, external=True)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        t0.record()
        for c in calls:
            txl.mem_update(mems[c["n"]], c["h"])
        t1.record()
    times = []
    for _ in range(reps):
        g.replay()
        torch.cuda.synchronize()
        times.append(t0.elapsed_time(t1) / len(calls))
    txl.check_status()
    return statistics.median(times)


def time_longmem_rolls(dev, stream, peaks, n_sets=6, reps=5):
    """The Tail_M roll of the long-memory configuration (B=8, L=128, M=3200,
    d=1024, bf16: 52.4 MB read + 52.4 MB written per roll), measured where its
    HBM target is quoted.  ``n_sets`` distinct (memory, hidden state) pairs
    (6 x 54.5 MB, well beyond the 126 MB L2) are rolled in rotation, 4 passes
    over the sets in one CUDA graph, so every roll reads memory that the L2
    no longer holds and its writes must reach DRAM; events bracket the whole
    graph only."""
    import transformer_xl_relative_attn_gb300 as txl

    wl = W.WORKLOADS["longmem3200_bf16"]
    B, L, M, d = wl.B, wl.L, wl.M, wl.d
    g = torch.Generator(device="cpu").manual_seed(29)
    mems = [torch.randn(B, M, d, generator=g).to(device=dev, dtype=torch.bfloat16) for _ in range(n_sets)]
    hids = [torch.randn(B, L, d, generator=g).to(device=dev, dtype=torch.bfloat16) for _ in range(n_sets)]
    passes = 4
    t0 = torch.cuda.Event(enable_timing=True, external=True)
    t1 = torch.cuda.Event(enable_timing=True, external=True)
    with torch.cuda.stream(stream):
        for m, h in zip(mems, hids):
            txl.mem_update(m, h, stream=stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        t0.record()
        for _ in range(passes):
            for m, h in zip(mems, hids):
                txl.mem_update(m, h)
        t1.record()
    times = []
    for _ in range(reps):
        graph.replay()
        torch.cuda.synchronize()
        times.append(t0.elapsed_time(t1) / (passes * n_sets))
    txl.check_status()
    ms = statistics.median(times)
    nbytes = wl.mem_update_bytes()
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    gbs = nbytes / (ms * 1e-3) / 1e9
    del mems, hids
    return {
        "kernel": "tail_chain_kernel", "workload": wl.name, "bound": "hbm",
        "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4),
        "peak_source": "hbm_gbs (measured copy bandwidth)",
        "bytes_per_launch": nbytes, "avg_launch_ms": round(ms, 5),
        "measured": f"{passes} passes over {n_sets} distinct memories (6 x 54.5 MB > L2) in one CUDA "
                    f"graph, events around the graph only; median of {reps} replays",
    }


def measure_e2e(args, wl, calls, stream, side, mems, rks, u, vb, scratch, flops_step, ws):
    """Same metric end to end through the public API: each step copies every
    input of the step from pinned host memory (q, k, v and the layer input h
    of every call) and reads every attention output back.  Copies run on
    their own streams and overlap the calls: call i starts once its inputs
    arrived, its output leaves once it is written; the next step's copies
    into a buffer wait until this step is done with it."""
    import transformer_xl_relative_attn_gb300 as txl

    ins = [[(c[x], c[x].cpu().pin_memory()) for x in ("q", "k", "v", "h")] for c in calls]
    outs = [(c["out"], torch.empty(c["out"].shape, dtype=c["out"].dtype).pin_memory()) for c in calls]
    h2d = sum(d.numel() * d.element_size() for call in ins for d, _ in call)
    d2h = sum(d.numel() * d.element_size() for d, _ in outs)
    steps = max(3, min(args.steps, 10))
    dev = stream.device
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    n_calls = len(calls)

    def one():
        arrived = [torch.cuda.Event() for _ in range(n_calls)]
        written = [torch.cuda.Event() for _ in range(n_calls)]
        rolled = {}
        with torch.cuda.stream(up):
            for i in range(n_calls):
                for d, hbuf in ins[i]:
                    d.copy_(hbuf, non_blocking=True)
                arrived[i].record(up)
        for i, c in enumerate(calls):
            n = c["n"]
            stream.wait_event(arrived[i])
            if n in rolled:
                stream.wait_event(rolled[n])
            ready = torch.cuda.Event()
            ready.record(stream)
            if scratch is None:
                txl.attn_fwd(c["q"], c["k"], c["v"], rks[n], u, vb, wl.scale, out=c["out"], stream=stream)
            else:
                txl.attn_fwd_ws(c["q"], c["k"], c["v"], rks[n], u, vb, scratch, wl.scale,
                                out=c["out"], stream=stream)
            written[i].record(stream)
            side.wait_event(ready)
            txl.mem_update(mems[n], c["h"], stream=side)
            rolled[n] = torch.cuda.Event()
            rolled[n].record(side)
            down.wait_event(written[i])
            with torch.cuda.stream(down):
                outs[i][1].copy_(outs[i][0], non_blocking=True)
        # the next step's copies overwrite these inputs and outputs
        for st in (stream, side, down):
            ev = torch.cuda.Event()
            ev.record(st)
            up.wait_event(ev)
            stream.wait_event(ev)

    one()
    torch.cuda.synchronize()
    barrier(ws)
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    torch.cuda.synchronize()
    el = reduce_max(time.perf_counter() - t0, ws)
    return {"value": round(ws * flops_step * steps / el / 1e12, 3), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": round(1e3 * el / steps, 3)}


def build_stack(wl, dev, stream):
    """An AttnStack of the workload's layers with the library's own
    projections: W_q, W_k, W_v stacked in the nn.Linear layout, r_k of every
    layer projected once by txl_r_proj from the sinusoid of distances
    M+L-1 .. 0, layer 0's memory in rows, the others in heads.  When L < M
    the memories are ring buffers (each segment writes L rows instead of
    moving M).  The rolls run on a second stream, overlapping the attention."""
    import transformer_xl_relative_attn_gb300 as txl
    bf = torch.bfloat16
    p = W.make_params(wl)
    H = wl.H
    with torch.cuda.stream(stream):
        w_qkv = [torch.cat([lw.W_q.t(), lw.W_k.t(), lw.W_v.t()]).contiguous().to(dev, bf) for lw in p.layers]
        emb = W.sinusoid(torch.arange(wl.M + wl.L - 1, -1, -1), wl.d).to(dev, bf)
        r_k = [txl.r_proj(emb, lw.W_r.t().contiguous().to(dev, bf), H, stream=stream) for lw in p.layers]
        u = [p.u.to(dev, bf)] * wl.layers
        vb = [p.v.to(dev, bf)] * wl.layers
        m0 = W.initial_memories(wl)
        mems = [m0[0].to(dev, bf)] + [W._split_heads(m, H).to(dev, bf) for m in m0[1:]]
    stream.synchronize()
    ring = wl.L < wl.M and wl.L % 128 == 0 and wl.M % 128 == 0
    return txl.AttnStack(w_qkv, r_k, u, vb, mems, wl.scale, H, wl.L, stream=stream, ring=ring,
                         mem_stream=torch.cuda.Stream(device=dev))


def measure_e2e_stack(args, wl, dev, flops_step, ws):
    """The metric end to end through the segment-level public API
    (AttnStack.run_segment: projections, Tail_M rolls and attention of every
    layer in libtxl.so).  Each step copies every segment's layer-0 hidden
    states [B, L, d] from pinned host memory and reads every segment's last
    attention output back; segment s+1's upload overlaps segment s's layers
    and segment s's download overlaps segment s+1's.  The step's work is the
    bench step's 36 attention calls and rolls plus the 36 projections; the
    value counts the attention FLOPs only."""
    import transformer_xl_relative_attn_gb300 as txl
    stream = torch.cuda.Stream(device=dev)
    stack = build_stack(wl, dev, stream)
    bf = torch.bfloat16
    S = wl.segments
    h_host = [W.segment_input(wl, s).to(bf).pin_memory() for s in range(S)]
    h_dev = [torch.empty(h.shape, dtype=bf, device=dev) for h in h_host]
    o_shape = (wl.B, wl.H, wl.L, wl.dh)
    o_dev = [torch.empty(o_shape, dtype=bf, device=dev) for _ in range(S)]
    o_host = [torch.empty(o_shape, dtype=bf).pin_memory() for _ in range(S)]
    h2d = sum(h.numel() * h.element_size() for h in h_host)
    d2h = sum(o.numel() * o.element_size() for o in o_host)
    steps = max(3, min(args.steps, 10))
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def one():
        arrived = [torch.cuda.Event() for _ in range(S)]
        with torch.cuda.stream(up):
            for s in range(S):
                h_dev[s].copy_(h_host[s], non_blocking=True)
                arrived[s].record(up)
        for s in range(S):
            stream.wait_event(arrived[s])
            stack.run_segment(h_dev[s], out=o_dev[s])
            written = torch.cuda.Event()
            written.record(stream)
            down.wait_event(written)
            with torch.cuda.stream(down):
                o_host[s].copy_(o_dev[s], non_blocking=True)
        # the next step's copies overwrite these buffers
        for st in (stream, down):
            ev = torch.cuda.Event()
            ev.record(st)
            up.wait_event(ev)
            stream.wait_event(ev)

    one()
    torch.cuda.synchronize()
    txl.check_status()
    barrier(ws)
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    torch.cuda.synchronize()
    el = reduce_max(time.perf_counter() - t0, ws)
    txl.check_status()
    return {"value": round(ws * flops_step * steps / el / 1e12, 3), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": round(1e3 * el / steps, 3),
            "tokens_per_s": round(ws * wl.B * wl.L * S * steps / el, 1),
            "api": "AttnStack.run_segment per segment (txl_qkv_proj_ring, txl_mem_update or "
                   "txl_mem_ring_push, txl_attn_fwd per layer); host hidden states in, last layer's "
                   "attention output out",
            "memory": "ring buffer" if stack.ring else "Tail_M copy"}


def measure_decoder(args, wl, dev, flops_step, ws, d_inner_mult=4):
    """Full decoder layers (DecoderStack, post-norm: attention, o_net,
    LayerNorm, feed-forward with d_inner = 4 d, LayerNorm) over the same
    segments, end to end with host I/O as in measure_e2e_stack.  Reports
    tokens/s and the attention TFLOP/s that this step sustains."""
    import transformer_xl_relative_attn_gb300 as txl
    bf = torch.bfloat16
    stream = torch.cuda.Stream(device=dev)
    d, H, L, M = wl.d, wl.H, wl.L, wl.M
    di = d_inner_mult * d
    g = torch.Generator().manual_seed(7)

    def n(*shape, std):
        return torch.empty(shape).normal_(0.0, std, generator=g).to(dev, bf)

    with torch.cuda.stream(stream):
        layers = [{"w_qkv": n(3 * d, d, std=0.02), "w_o": n(d, d, std=0.02),
                   "ln1_g": torch.ones(d, dtype=bf, device=dev), "ln1_b": torch.zeros(d, dtype=bf, device=dev),
                   "w1": n(di, d, std=0.02), "b1": n(di, std=0.02), "w2": n(d, di, std=0.02),
                   "b2": n(d, std=0.02), "ln2_g": torch.ones(d, dtype=bf, device=dev),
                   "ln2_b": torch.zeros(d, dtype=bf, device=dev)} for _ in range(wl.layers)]
        emb = W.sinusoid(torch.arange(M + L - 1, -1, -1), d).to(dev, bf)
        r_k = [txl.r_proj(emb, n(d, d, std=0.02), H, stream=stream) for _ in range(wl.layers)]
        u = [n(H, wl.dh, std=0.02)] * wl.layers
        vb = [n(H, wl.dh, std=0.02)] * wl.layers
        mems = [n(wl.B, M, d, std=1.0) for _ in range(wl.layers)]
    stream.synchronize()
    stack = txl.DecoderStack(layers, r_k, u, vb, mems, wl.scale, H, L, stream=stream)
    S = wl.segments
    h_host = [W.segment_input(wl, s).to(bf).pin_memory() for s in range(S)]
    h_dev = [torch.empty(h.shape, dtype=bf, device=dev) for h in h_host]
    o_dev = [torch.empty(h.shape, dtype=bf, device=dev) for h in h_host]
    o_host = [torch.empty(h.shape, dtype=bf).pin_memory() for h in h_host]
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    steps = max(3, min(args.steps, 10))

    def one():
        arrived = [torch.cuda.Event() for _ in range(S)]
        with torch.cuda.stream(up):
            for s in range(S):
                h_dev[s].copy_(h_host[s], non_blocking=True)
                arrived[s].record(up)
        for s in range(S):
            stream.wait_event(arrived[s])
            stack.run_segment(h_dev[s], out=o_dev[s])
            written = torch.cuda.Event()
            written.record(stream)
            down.wait_event(written)
            with torch.cuda.stream(down):
                o_host[s].copy_(o_dev[s], non_blocking=True)
        for st in (stream, down):
            ev = torch.cuda.Event()
            ev.record(st)
            up.wait_event(ev)
            stream.wait_event(ev)

    one()
    torch.cuda.synchronize()
    txl.check_status()
    barrier(ws)
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    torch.cuda.synchronize()
    el = reduce_max(time.perf_counter() - t0, ws)
    txl.check_status()
    # dense flops of the layer besides attention: qkv, o_net, two FF layers
    T = wl.B * L
    other = 2 * wl.layers * S * (T * d * d + wl.B * (M + L) * 2 * d * d + T * d * d + 2 * T * d * di)
    return {"ms_per_step": round(1e3 * el / steps, 3),
            "tokens_per_s": round(ws * wl.B * L * S * steps / el, 1),
            "attn_tflops": round(ws * flops_step * steps / el / 1e12, 3),
            "all_matmul_tflops": round(ws * (flops_step + other) * steps / el / 1e12, 3),
            "d_inner": di, "norm": "post", "steps": steps,
            "api": "DecoderStack.run_segment per segment; host hidden states in, last layer output out"}


def time_backward(wl, calls, rks, u, vb, dev, peak_tf=None, peak_src=""):
    """txl_attn_bwd_ws on the workload's first call (bf16 inputs, fp32
    gradients), timed alone with CUDA events: 2 warm-up, 10 timed calls, the
    caller's workspace and gradient buffers reused.  Algorithmic work 12 d_h
    FLOPs per visible pair (the six contractions dV, dP, dq content, dq
    position, dk, dR; the recomputed scores are not counted).  The tensor-core
    passes run where they apply (bf16, d_h = 64): the peak is then the bf16
    tensor peak; otherwise the CUDA-core kernel against the fp32 FMA rate of
    the SMs at their maximum clock (152 x 128 FMA/clk x 2 FLOP x 2.07 GHz)."""
    import transformer_xl_relative_attn_gb300 as txl
    c = calls[0]
    g = torch.randn(c["q"].shape, generator=torch.Generator().manual_seed(0)).to(dev, c["q"].dtype)
    need = txl.attn_bwd_workspace_bytes(wl.B, wl.H, wl.L, wl.M, wl.dh, c["q"].dtype, device=dev)
    ws = torch.empty(need, dtype=torch.uint8, device=dev) if need else None
    args = (c["q"], c["k"], c["v"], rks[0], u, vb, g, wl.scale)
    grads = txl.attn_bwd(*args, workspace=ws)
    for _ in range(2):
        txl.attn_bwd(*args, workspace=ws, grads=grads)
    torch.cuda.synchronize()
    n = 10 if need else 3
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n):
        txl.attn_bwd(*args, workspace=ws, grads=grads)
    e1.record()
    torch.cuda.synchronize()
    txl.check_status()
    ms = e0.elapsed_time(e1) / n
    flops = 12 * wl.dh * wl.B * wl.H * wl.visible_pairs()
    tf = flops / (ms * 1e-3) / 1e12
    if need:
        kern = "attn_tc_bf16_kernel (the forward with lse) + attn_bwd_prep_kernel + attn_bwd_q_kernel + attn_bwd_kv_kernel"
        bound, peak, psrc = "tensor", peak_tf, f"bf16_tflops, burst ({peak_src})"
    else:
        kern = "attn_bwd_tiled_kernel" if wl.dh <= 64 else "attn_bwd_simt_kernel"
        bound, peak, psrc = "alu", 152 * 128 * 2 * 2.07e9 / 1e12, "derived: fp32 FMA units x max SM clock"
    res = {"kernel": kern, "ms": round(ms, 4), "tflops": round(tf, 3), "bound": bound, "peak": round(peak, 1),
           "frac": round(tf / peak, 4), "peak_source": psrc, "flops": flops,
           "measured": f"the workload's first call alone, CUDA events, {n} calls, whole backward (all launches, "
                       "the forward and its lse recomputed inside)"}
    if need and wl.dh == 64:
        # the same gradients from the forward's saved state (out and the rows'
        # log2-sum-exp, as a training forward keeps them): no recomputed forward
        out, lse = txl.attn_fwd_lse(c["q"], c["k"], c["v"], rks[0], u, vb, scale=wl.scale)
        for _ in range(2):
            txl.attn_bwd(*args, workspace=ws, grads=grads, out=out, lse=lse)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(n):
            txl.attn_bwd(*args, workspace=ws, grads=grads, out=out, lse=lse)
        e1.record()
        torch.cuda.synchronize()
        txl.check_status()
        ms2 = e0.elapsed_time(e1) / n
        tf2 = flops / (ms2 * 1e-3) / 1e12
        res["from_saved_state"] = {
            "entry": "txl_attn_bwd_saved (out and lse from txl_attn_fwd_lse)",
            "kernel": "attn_bwd_prep_kernel + attn_bwd_q_kernel + attn_bwd_kv_kernel",
            "ms": round(ms2, 4), "tflops": round(tf2, 3), "frac": round(tf2 / peak, 4)}
    return res


def cpu_baseline_and_parity(wl, calls, rks, u, vb):
    """Times the fp64 oracle on the first call of the workload (segment 0,
    layer 0, every (batch row, head) pair) on all host cores, and re-checks
    that call's GPU output against it."""
    import oracle
    c = calls[0]
    host = [t.cpu() for t in (c["q"], c["k"], c["v"], rks[0], u, vb)]
    t0 = time.perf_counter()
    ref = oracle.attn(*host, wl.scale)
    el = time.perf_counter() - t0
    got = c["out"].float().cpu().double().numpy()
    err = float(np.abs(got - ref).max())
    tol = 1e-2 * float(np.abs(ref).max()) + 1e-3
    cb = {"value": round(wl.attn_flops() / el / 1e12, 6), "unit": "TFLOP/s",
          "cores": oracle.num_cores(), "kind": "oracle",
          "sample": f"one txl_attn_fwd call of {wl.name} (segment 0, layer 0, all {wl.B * wl.H} "
                    f"(b,h) pairs), fp64, {el:.2f} s wall"}
    par = {"call": "segment 0, layer 0", "max_abs_err": err, "tol": tol, "ok": err <= tol}
    return cb, par


# --------------------------------------------------------------------- reference arm
def run_reference(args, wl: W.Workload):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    ci, _, _ = W.first_call_inputs(wl)
    n = wl.B * wl.H
    per_pair_flops = 6 * wl.dh * wl.visible_pairs()
    rng = np.random.default_rng(0)
    # size one step to about 0.2-0.5 s of oracle time on this host
    k_pairs = max(1, min(n, 2 * oracle.num_cores()))
    host = (ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb)

    def one():
        pairs = rng.choice(n, size=k_pairs, replace=False)
        oracle.attn(*host, ci.scale, pairs=pairs)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    el = time.perf_counter() - t0
    value = per_pair_flops * k_pairs * args.steps / el / 1e12
    sample = (f"{k_pairs} random (b,h) pairs of the first {wl.name} call per step "
              f"(of {n}), fp64 oracle")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * el / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "H": wl.H, "d_h": wl.dh, "L": wl.L, "M": wl.M},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.num_cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    wl = W.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
