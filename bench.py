#!/usr/bin/env python3
"""Throughput of the Llama decoder block forward on GB300, one JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-decode]

Headline workload: one Llama-3-8B-shaped block prefill, B=1, S=8192 (bf16, fp32 accumulation).
A step is one llama_block_forward call over the 8192 tokens (RMSNorm, fused QKV+RoPE+KV write,
causal GQA attention, O projection + residual, RMSNorm, gate/up + SiLU*mul, down + residual), bf16
input and weights, output in fp32 (LLAMA_Y_F32: the residual stream a stack hands on).
`decode` reports the 32-layer batch-64 decode step against 8192 cached positions
(llama_stack_decode_step, replayed as a CUDA graph).  Under torchrun every rank runs its own
replica (the block has no exchange step); value = all ranks' tokens / max rank time.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "block-forward tokens/s (prefill & decode) at 1 GB300; % of TC/HBM roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def sources_sha(files) -> str:
    """Hash of the named kernel sources (file names under the package's csrc/)."""
    import hashlib
    h = hashlib.sha256()
    for name in sorted(files):
        h.update(name.encode())
        with open(os.path.join(ROOT, "llama_decoder_block_fwd_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def kernel_traffic(role: str):
    """Measured DRAM bytes per launch of a kernel role from profiles/traffic.json, or None when that
    kernel's sources have changed since the capture."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            k = json.load(f).get("kernels", {}).get(role)
        if k is None or sources_sha(k["sources"]) != k["sha"]:
            return None
    except Exception:
        return None
    return k["bytes_per_launch"]


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return FALLBACK_PEAKS, "fallback"


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device: int):
        import torch
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            cmd.insert(1, f"--id=GPU-{uuid}")
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        return parse_clocks(out)


def parse_clocks(out: str) -> dict:
    """The clocks record of the timed region from nvidia-smi's CSV lines (ClockSampler.FIELDS, no
    header, no units): median SM clock of the samples under load (at least half the highest), the
    maximum SM clock, and every throttle reason seen active in any sample."""
    sm, smax, reasons = [], [], set()
    for line in out.strip().splitlines():
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm.append(float(parts[1]))
            smax.append(float(parts[2]))
        except ValueError:
            continue
        for name, val in zip(ClockSampler.NAMES, parts[5:9]):
            if val.lower() == "active":
                reasons.add(name)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
    hi = [s for s in sm if s >= 0.5 * max(sm)]   # samples under load
    return {"sm_mhz": statistics.median(hi), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
            "samples": len(sm)}


# ----------------------------------------------------------------------------- helpers
def dist_setup(backend: str = "nccl"):
    """One process per GPU (torchrun's RANK / LOCAL_RANK / WORLD_SIZE).  Every rank runs an
    independent replica of the step on its own synthetic data: the block has no exchange step,
    so the process group carries only the barriers and the max-over-ranks of the timings."""
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    cuda = backend == "nccl"
    if cuda:
        torch.cuda.set_device(local if world > 1 else 0)
    if world > 1:
        import torch.distributed as dist
        if cuda:
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    return world, rank, local


def barrier(world, cuda: bool = True):
    if cuda:
        import torch
        torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    if cuda:
        import torch
        torch.cuda.synchronize()


def max_over_ranks(world, v: float, device: str = "cuda") -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(world: int, units_per_rank: float, ms_max: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest rank's time."""
    return world * units_per_rank / (ms_max / 1e3)


def prefill_flops(wl):
    """Algorithmic FLOPs of one block forward: 2mnp for the seven projections, causal attention
    (QK^T and PV over the visible keys only: 4 * n_q * hd * S(S+1)/2 per sequence)."""
    T = wl.B * wl.S
    hq, hkv = wl.n_q * wl.head_dim, wl.n_kv * wl.head_dim
    return {
        "gemm_tc_qkv": 2.0 * T * wl.d_model * (hq + 2 * hkv),
        "gemm_tc_resid": 2.0 * T * (hq * wl.d_model + wl.d_ff * wl.d_model),
        "gemm_tc_swiglu": 2.0 * T * wl.d_model * 2 * wl.d_ff,
        "attn": 4.0 * wl.n_q * wl.head_dim * wl.B * wl.S * (wl.S + 1) / 2,
    }


def decode_bytes(wl, kv_elem_bytes=2):
    """Algorithmic HBM bytes of one decode step: every cached K/V read once (kv_elem_bytes per
    element), every bf16 weight read once, the new K/V written, inputs read and logits written."""
    L, B, t = wl.n_layers, wl.B, wl.t_cache
    row = wl.n_kv * wl.head_dim
    kv_read = L * B * (t + 1) * row * 2 * kv_elem_bytes
    hq = wl.n_q * wl.head_dim
    layer_w = (wl.d_model * (hq + 2 * row) + hq * wl.d_model + 3 * wl.d_model * wl.d_ff + 2 * wl.d_model) * 2
    return {
        "kv_read": kv_read,
        "weights": L * layer_w,
        "lm_head": wl.vocab * wl.d_model * 2 + wl.d_model * 2,
        "kv_append": L * B * row * 2 * kv_elem_bytes,
        "logits": B * wl.vocab * 4,
        "input": B * wl.d_model * 2,
    }


# ----------------------------------------------------------------------------- our arm
def bench_mha_prefill(args, world):
    """The LLaMA-7B (MHA, n_kv = n_q) block prefill, B4 S2048: device-timed steps only."""
    import torch

    import llama_decoder_block_fwd_gb300 as L
    from synth import configs as C
    from synth import workloads as W

    wl = C.LLAMA_7B_MHA_PREFILL
    T = wl.B * wl.S
    w = W.device_layer(wl)
    x = W.device_x(wl).reshape(T, wl.d_model)
    y = torch.empty(x.shape, dtype=torch.float32, device="cuda")   # fp32 residual stream out
    ws = torch.empty(L.llama_workspace_bytes(L.OP_BLOCK_FORWARD, wl.dims, wl.dtype), dtype=torch.uint8,
                     device="cuda")
    bw = L.block_weights(w)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        L.llama_block_forward(wl.dims, wl.dtype | L.Y_F32, bw, x, y, 0, None, None, 0, ws, stream)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        L.llama_block_forward(wl.dims, wl.dtype | L.Y_F32, bw, x, y, 0, None, None, 0, ws, stream)
    e1.record(stream)
    barrier(world)
    if L.llama_get_device_status() != 0:
        raise RuntimeError("device status word set during the MHA prefill")
    ms = max_over_ranks(world, e0.elapsed_time(e1)) / args.steps
    pk, pk_src = peaks()
    hq = wl.n_q * wl.head_dim
    flops = 2.0 * T * (wl.d_model * (hq + 2 * wl.n_kv * wl.head_dim) + hq * wl.d_model + 3 * wl.d_model * wl.d_ff) \
        + 4.0 * wl.n_q * wl.head_dim * wl.B * wl.S * (wl.S + 1) / 2
    out = {"workload": wl.name, "value": aggregate_rate(world, T, ms), "unit": "tokens/s", "ms_per_step": ms,
           "flops_per_step": flops, "block_tflops": flops / (ms / 1e3) / 1e12,
           "block_tc_frac": flops / (ms / 1e3) / 1e12 / pk["bf16_tflops"], "peak_source": f"{pk_src} bf16 burst"}
    del w, x, y, ws
    torch.cuda.empty_cache()
    return out


class L2Flush:
    """Evicts L2 between timed calls: a 256 MB write, then a 256 MB read, so that L2 (129 MB)
    holds neither the timed call's inputs nor dirty lines whose write-back would land inside the
    timed call.  The ~80 us of device work also covers the host's launch latency of the call."""
    what = "flushed before every call (256 MB written, then 256 MB read)"

    def __init__(self):
        import torch
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        self.r = torch.ones(64 << 20, dtype=torch.int32, device="cuda")

    def __call__(self):
        self.w.fill_(1)
        self.r.sum()


def bench_sample(args, world):
    """Next-token choice for the decode batch: 64 rows of 128256 fp32 logits, temperature 0.8,
    top-k 50, top-p 0.95.  L2 is flushed (L2Flush) before every timed call."""
    import numpy as np
    import torch

    import llama_decoder_block_fwd_gb300 as L
    from synth import F32, TID_LOGITS
    from synth import configs as C
    from synth import workloads as W

    wl = C.LLAMA3_8B_DECODE
    z = W.device_tensor(F32, (wl.B, wl.vocab), wl.seed, TID_LOGITS, 0.0, 2.5)
    u = torch.from_numpy(np.random.default_rng(wl.seed).random(wl.B).astype(np.float32)).cuda()
    tok = torch.empty(wl.B, dtype=torch.int32, device="cuda")
    flush = L2Flush()
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        L.llama_sample(z, 0.8, 50, 0.95, u, tok)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    for a, b in ev:
        flush()
        a.record(stream)
        L.llama_sample(z, 0.8, 50, 0.95, u, tok)
        b.record(stream)
    barrier(world)
    ms = max_over_ranks(world, sum(a.elapsed_time(b) for a, b in ev) / args.steps)
    nbytes = z.numel() * 4
    out = {"workload": f"{wl.B} x {wl.vocab} fp32 logits, T 0.8, top-k 50, top-p 0.95", "us_per_call": ms * 1e3,
           "rows_per_s": aggregate_rate(world, wl.B, ms), "logits_gbs": nbytes / (ms / 1e3) / 1e9,
           "l2": L2Flush.what}
    del z, u, tok, flush
    torch.cuda.empty_cache()
    return out


def bench_rmsnorm(args, world):
    """Standalone llama_rmsnorm on the 8B block's prefill activations: 8192 x 4096 bf16 rows in,
    bf16 rows out, bf16 gains.  L2 is flushed (L2Flush) before every timed call."""
    import torch

    import llama_decoder_block_fwd_gb300 as L
    from synth import configs as C
    from synth import workloads as W

    wl = C.LLAMA3_8B_PREFILL
    if args.rmsnorm_rows != wl.S:
        wl = dataclasses.replace(wl, S=args.rmsnorm_rows, name=f"{wl.name}-rows{args.rmsnorm_rows}")
    T = wl.B * wl.S
    x = W.device_x(wl).reshape(T, wl.d_model)
    g = W.device_layer(wl)["attn_norm_g"]
    y = torch.empty_like(x)
    dims = (wl.B, wl.S, wl.d_model, wl.n_q, wl.n_kv, wl.head_dim, wl.d_ff, wl.theta_base, wl.eps)
    flush = L2Flush()
    stream = torch.cuda.current_stream()
    # warm-up: at least W calls and a quarter second of them (a GPU fresh from idle ran its first
    # few milliseconds of calls up to 20% slower)
    t0, n = time.perf_counter(), 0
    while n < args.warmup or time.perf_counter() - t0 < 0.25:
        flush()
        L.llama_rmsnorm(dims, wl.dtype, x, g, y, stream)
        n += 1
    steps = max(args.steps, 100)   # ~40 ms of calls with their flushes
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(world)
    for a, b in ev:
        flush()
        a.record(stream)
        L.llama_rmsnorm(dims, wl.dtype, x, g, y, stream)
        b.record(stream)
    barrier(world)
    if L.llama_get_device_status() != 0:
        raise RuntimeError("device status word set during the RMSNorm line")
    ms = max_over_ranks(world, sum(a.elapsed_time(b) for a, b in ev) / steps)
    pk, pk_src = peaks()
    nbytes = x.numel() * 2 + y.numel() * 2 + g.numel() * 2
    gbs = nbytes / (ms / 1e3) / 1e9
    out = {"workload": f"llama_rmsnorm {T} x {wl.d_model} bf16", "us_per_call": ms * 1e3, "bytes_per_call": nbytes,
           "calls_timed": steps, "warmup_calls": n,
           "roofline": {"bound": "hbm", "kernel": "rmsnorm_stream", "achieved": gbs, "peak": pk["hbm_gbs"],
                        "unit": "GB/s", "frac": gbs / pk["hbm_gbs"], "peak_source": f"{pk_src} hbm",
                        "traffic": kernel_traffic("rmsnorm_stream") if T == 8192 else None},
           "l2": L2Flush.what}
    del x, g, y, flush
    torch.cuda.empty_cache()
    return out


def bench_prefill(args, world, rank):
    import torch

    import llama_decoder_block_fwd_gb300 as L
    from synth import configs as C
    from synth import workloads as W

    wl = C.LLAMA3_8B_PREFILL
    if args.prefill_seq != wl.S:   # smaller sequence for sizing profiler captures
        import dataclasses
        wl = dataclasses.replace(wl, S=args.prefill_seq, name=f"{wl.name}-S{args.prefill_seq}")
    T = wl.B * wl.S
    w = W.device_layer(wl)
    x = W.device_x(wl).reshape(T, wl.d_model)
    y = torch.empty(x.shape, dtype=torch.float32, device="cuda")   # fp32 residual stream out
    ws = torch.empty(L.llama_workspace_bytes(L.OP_BLOCK_FORWARD, wl.dims, wl.dtype), dtype=torch.uint8,
                     device="cuda")
    bw = L.block_weights(w)
    stream = torch.cuda.current_stream()

    def step():
        L.llama_block_forward(wl.dims, wl.dtype | L.Y_F32, bw, x, y, 0, None, None, 0, ws, stream)

    for _ in range(args.warmup):
        step()
    barrier(world)
    if L.llama_get_device_status() != 0:
        raise RuntimeError("device status word set during warm-up")
    # the step time comes from K steps with nothing between the launches; the per-kernel durations
    # (roofline, kernel shares) from a second pass of K steps with an event pair around each launch,
    # which adds small gaps of its own
    clocks = ClockSampler(torch.cuda.current_device())
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    barrier(world)
    clk = clocks.stop()
    ms_total = max_over_ranks(world, e0.elapsed_time(e1))
    # a second, longer region (about one second of back-to-back steps) for the rate under the
    # power cap, reported beside the headline against the sustained bf16 peak
    n_sus = max(args.steps, int(1000.0 / max(ms_total / args.steps, 1e-3)) + 1)
    barrier(world)
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for _ in range(n_sus):
        step()
    s1.record(stream)
    barrier(world)
    ms_sus = max_over_ranks(world, s0.elapsed_time(s1)) / n_sus
    L.llama_profile_read()            # clear
    L.llama_profile_enable(True)
    barrier(world)
    for _ in range(args.steps):
        step()
    barrier(world)
    L.llama_profile_enable(False)
    prof = L.llama_profile_read()
    if L.llama_get_device_status() != 0:
        raise RuntimeError("device status word set during the timed region")

    # end to end: pinned host x -> device, block, device y -> pinned host, every step.  The copies
    # run on their own streams with two device buffers each, so step i+1's input copy and step
    # i-1's output copy overlap step i's block; the timed region still holds every step's copies.
    xh = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    xh.copy_(x)
    yh = [torch.empty(y.shape, dtype=y.dtype, pin_memory=True) for _ in range(2)]
    xd = [torch.empty_like(x) for _ in range(2)]
    yd = [torch.empty_like(y) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    in_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(n, start_ev=None, end_ev=None):
        if start_ev is not None:
            start_ev.record(stream)
            s_in.wait_event(start_ev)
        for i in range(n):
            k = i & 1
            if i >= 2:
                s_in.wait_event(comp_done[k])      # step i-2 has read xd[k]
            with torch.cuda.stream(s_in):
                xd[k].copy_(xh, non_blocking=True)
                in_done[k].record(s_in)
            stream.wait_event(in_done[k])
            if i >= 2:
                stream.wait_event(out_done[k])     # step i-2's result has left yd[k]
            L.llama_block_forward(wl.dims, wl.dtype | L.Y_F32, bw, xd[k], yd[k], 0, None, None, 0, ws, stream)
            comp_done[k].record(stream)
            s_out.wait_event(comp_done[k])
            with torch.cuda.stream(s_out):
                yh[k].copy_(yd[k], non_blocking=True)
                out_done[k].record(s_out)
        stream.wait_event(out_done[(n - 1) & 1])
        if n >= 2:
            stream.wait_event(out_done[(n - 2) & 1])
        if end_ev is not None:
            end_ev.record(stream)

    e2e_run(2)
    torch.cuda.synchronize()
    barrier(world)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_run(args.steps, f0, f1)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(world, f0.elapsed_time(f1))
    e2e_same = bool(torch.equal(yh[(args.steps - 1) & 1], y.cpu()))   # bit-identical to the resident step

    pk, pk_src = peaks()
    flops = prefill_flops(wl)
    step_flops = sum(flops.values())
    kernels = {}
    launches = 0
    for name, (n, ms) in prof.items():
        kernels[name] = {"launches": n, "ms_per_step": ms / args.steps, "share": ms / max(sum(v[1] for v in prof.values()), 1e-9)}
        launches += n
    dom = max(prof.items(), key=lambda kv: kv[1][1])[0] if prof else None
    dom_key = "attn" if dom and dom.startswith("attn") else dom
    dom_flops = flops.get(dom_key, 0.0)
    dom_ms = prof[dom][1] if dom else 0.0
    timed_s = ms_total / 1e3
    peak_tf = pk["bf16_tflops_sustained"] if timed_s > 1.0 else pk["bf16_tflops"]
    achieved = dom_flops * args.steps / (dom_ms / 1e3) / 1e12 if dom_ms > 0 else 0.0
    ms_step = ms_total / args.steps
    out = {
        "value": aggregate_rate(world, T, ms_step),
        "ms_per_step": ms_step,
        "clocks": clk,
        "e2e": {"value": aggregate_rate(world, T, e2e_ms / args.steps), "unit": "tokens/s",
                "h2d_bytes_per_step": x.numel() * x.element_size(),
                "d2h_bytes_per_step": y.numel() * y.element_size(),
                "copies": "pinned host buffers; H2D and D2H on their own streams, double-buffered, overlapping "
                          "the neighbouring steps' blocks",
                "result_equals_resident_step": e2e_same},
        "gpu_launches": launches,
        "roofline": {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": achieved / peak_tf, "traffic": kernel_traffic(dom) if wl.S == 8192 else None,
                     "peak_source": f"{pk_src} bf16 {'sustained' if timed_s > 1.0 else 'burst'}"},
        "block_tc_frac": step_flops / (ms_step / 1e3) / 1e12 / peak_tf,
        "block_tflops": step_flops / (ms_step / 1e3) / 1e12,
        "kernels": kernels,
        "config": prefill_config(wl, world, step_flops),
        "sustained": {"steps": n_sus, "timed_s": n_sus * ms_sus / 1e3, "ms_per_step": ms_sus,
                      "value": aggregate_rate(world, T, ms_sus), "block_tflops": step_flops / (ms_sus / 1e3) / 1e12,
                      "block_tc_frac": step_flops / (ms_sus / 1e3) / 1e12 / pk["bf16_tflops_sustained"],
                      "peak_source": f"{pk_src} bf16 sustained"},
    }
    del w, x, y, ws, xh, yh, xd
    torch.cuda.empty_cache()
    return out


def bench_decode(args, world, rank, kv8=False, seqs=None, cached=None):
    """One 32-layer decode step for 64 sequences holding 8192 cached positions (or `seqs`
    sequences holding `cached` positions).  kv8: the cache holds E4M3 codes with per-head scales
    (made from the same synthetic values by llama_kv_quantize) instead of bf16."""
    import numpy as np
    import torch

    import llama_decoder_block_fwd_gb300 as L
    from synth import configs as C
    from synth import workloads as W

    wl = C.LLAMA3_8B_DECODE
    if args.decode_layers != wl.n_layers:   # fewer layers for sizing profiler captures
        import dataclasses
        wl = dataclasses.replace(wl, n_layers=args.decode_layers, name=f"{wl.name}-L{args.decode_layers}")
    if seqs is not None:
        import dataclasses
        wl = dataclasses.replace(wl, B=seqs, t_cache=cached, name=f"llama3-8b-{wl.n_layers}L-decode-B{seqs}-T{cached}")
    cap = wl.t_cache + 1
    tensors = []
    layers = []
    for l in range(wl.n_layers):
        t = W.device_layer(wl, l)
        tensors.append(t)
        layers.append(L.block_weights(t))
    scales = None
    if kv8:
        scales = torch.full((wl.n_layers, 2, wl.n_kv), 0.03125, dtype=torch.float32, device="cuda")
        kc = torch.empty((wl.n_layers, wl.B, cap, wl.n_kv, wl.head_dim), dtype=torch.uint8, device="cuda")
        vc = torch.empty_like(kc)
        for l in range(wl.n_layers):
            for which, dst in (("k", kc), ("v", vc)):
                x = W.device_tensor(wl.dtype, (wl.B, cap, wl.n_kv, wl.head_dim), wl.seed, W.cache_tid(which, l),
                                    0.0, 1.0)
                L.llama_kv_quantize(x, scales[l, 0 if which == "k" else 1], dst[l])
                del x
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    else:
        kc, vc = W.device_caches(wl, cap)
    final_g, w_lm = W.device_final(wl)
    x = W.device_x_emb(wl)
    logits = torch.empty((wl.B, wl.vocab), dtype=torch.float32, device="cuda")
    ws = torch.empty(L.llama_workspace_bytes(L.OP_STACK_DECODE_STEP, wl.dims, wl.dtype, wl.n_layers, wl.vocab, cap),
                     dtype=torch.uint8, device="cuda")

    def step(stream=None):
        if kv8:
            L.llama_stack_decode_step_kv8(wl.dims, layers, final_g, w_lm, wl.vocab, x, kc, vc, scales, cap,
                                          wl.t_cache, logits, ws, stream)
        else:
            L.llama_stack_decode_step(wl.dims, wl.dtype, layers, final_g, w_lm, wl.vocab, x, kc, vc, cap, wl.t_cache,
                                      logits, ws, stream)

    # eager pass with per-launch events (per-kernel durations), then graph replay for the step time
    step()
    barrier(world)
    L.llama_profile_read()
    L.llama_profile_enable(True)
    nprof = max(2, min(args.steps, 5))
    for _ in range(nprof):
        step()
    L.llama_profile_enable(False)
    prof = L.llama_profile_read()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(args.warmup):
        g.replay()
    barrier(world)
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        g.replay()
    e1.record(stream)
    barrier(world)
    if L.llama_get_device_status() != 0:
        raise RuntimeError("device status word set during decode")
    ms = max_over_ranks(world, e0.elapsed_time(e1)) / args.steps
    pk, pk_src = peaks()
    nb = decode_bytes(wl, kv_elem_bytes=1 if kv8 else 2)
    step_bytes = sum(nb.values())
    kernels = {k: [n // nprof, round(t / nprof, 4)] for k, (n, t) in prof.items()}   # [launches, ms per step]
    attn = [k for k in prof if k.startswith("attn")]
    dom = max(prof.items(), key=lambda kv: kv[1][1])[0]
    out = {
        "workload": wl.name + ("-kv8" if kv8 else ""), "value": aggregate_rate(world, wl.B, ms), "unit": "tokens/s",
        "ms_per_step": ms, "bytes_per_step": step_bytes,
        "hbm_frac_step": step_bytes / (ms / 1e3) / 1e9 / pk["hbm_gbs"],
        "gpu_launches_per_step": sum(n for n, _ in prof.values()) // nprof,
        "kernels": kernels, "dominant_kernel": dom,
        "graph": "CUDA graph replay of one decode step",
        "l2": f"inputs larger than L2 ({step_bytes / 1e9:.0f} GB per step)",
    }
    if kv8:
        out["kv_cache"] = "E4M3 codes, per-(layer, K/V, head) fp32 scale 2^-5"
    if attn:
        a = attn[0]
        n, t = prof[a]
        per_launch_bytes = nb["kv_read"] / wl.n_layers
        achieved = per_launch_bytes / (t / n / 1e3) / 1e9
        out["roofline"] = {"bound": "hbm", "kernel": a, "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                           "frac": achieved / pk["hbm_gbs"], "traffic": kernel_traffic(a), "peak_source": f"{pk_src} hbm",
                           "algorithmic_bytes_per_launch": per_launch_bytes}
    del tensors, layers, kc, vc, final_g, w_lm, x, logits, ws, g, scales
    torch.cuda.empty_cache()
    return out


def bench_chunked_prefill(args, world):
    """Chunked prefill: the 8B block on 2048 new tokens at positions 6144..8191 of one sequence
    whose first 6144 positions are already in the cache (the call attends to them and appends its
    own K/V).  Each step rewrites the same cache rows with the same values."""
    import dataclasses

    import torch

    import llama_decoder_block_fwd_gb300 as L
    from synth import BF16, TID_KCACHE, TID_VCACHE
    from synth import configs as C
    from synth import workloads as W

    pos0, cap = 6144, 8192
    wl = dataclasses.replace(C.LLAMA3_8B_PREFILL, S=2048, name="llama3-8b-block-chunk-S2048-after-6144")
    T = wl.B * wl.S
    w = W.device_layer(wl)
    bw = L.block_weights(w)
    x = W.device_x(wl).reshape(T, wl.d_model)
    y = torch.empty(x.shape, dtype=torch.float32, device="cuda")   # fp32 residual stream out
    kc = W.device_tensor(BF16, (wl.B, cap, wl.n_kv, wl.head_dim), wl.seed, TID_KCACHE, 0.0, 1.0)
    vc = W.device_tensor(BF16, (wl.B, cap, wl.n_kv, wl.head_dim), wl.seed, TID_VCACHE, 0.0, 1.0)
    ws = torch.empty(L.llama_workspace_bytes(L.OP_BLOCK_FORWARD, wl.dims, wl.dtype), dtype=torch.uint8,
                     device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        L.llama_block_forward(wl.dims, wl.dtype | L.Y_F32, bw, x, y, pos0, kc, vc, cap, ws, stream)

    for _ in range(args.warmup):
        step()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    barrier(world)
    if L.llama_get_device_status() != 0:
        raise RuntimeError("device status word set during the chunked prefill")
    ms = max_over_ranks(world, e0.elapsed_time(e1)) / args.steps
    fl = prefill_flops(wl)
    fl["attn"] = 4.0 * wl.n_q * wl.head_dim * wl.B * (wl.S * pos0 + wl.S * (wl.S + 1) / 2)
    flops = sum(fl.values())
    pk, pk_src = peaks()
    out = {"workload": wl.name, "value": aggregate_rate(world, T, ms), "unit": "tokens/s", "ms_per_step": ms,
           "pos0": pos0, "flops_per_step": flops, "block_tflops": flops / (ms / 1e3) / 1e12,
           "block_tc_frac": flops / (ms / 1e3) / 1e12 / pk["bf16_tflops"], "peak_source": f"{pk_src} bf16 burst"}
    del w, bw, x, y, kc, vc, ws
    torch.cuda.empty_cache()
    return out


def bench_prefill_long(args, world):
    """The 8B block over one 32768-token sequence (RoPE base 5e5): causal attention is 38% of the
    FLOPs at this length."""
    import dataclasses

    import torch

    import llama_decoder_block_fwd_gb300 as L
    from synth import configs as C
    from synth import workloads as W

    wl = dataclasses.replace(C.LLAMA3_8B_PREFILL, S=32768, name="llama3-8b-block-prefill-B1-S32768")
    T = wl.B * wl.S
    w = W.device_layer(wl)
    bw = L.block_weights(w)
    x = W.device_x(wl).reshape(T, wl.d_model)
    y = torch.empty(x.shape, dtype=torch.float32, device="cuda")   # fp32 residual stream out
    ws = torch.empty(L.llama_workspace_bytes(L.OP_BLOCK_FORWARD, wl.dims, wl.dtype), dtype=torch.uint8,
                     device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        L.llama_block_forward(wl.dims, wl.dtype | L.Y_F32, bw, x, y, 0, None, None, 0, ws, stream)

    for _ in range(args.warmup):
        step()
    barrier(world)
    n = max(2, min(args.steps, 5))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        step()
    e1.record(stream)
    barrier(world)
    if L.llama_get_device_status() != 0:
        raise RuntimeError("device status word set during the long prefill")
    ms = max_over_ranks(world, e0.elapsed_time(e1)) / n
    fl = sum(prefill_flops(wl).values())
    pk, pk_src = peaks()
    out = {"workload": wl.name, "value": aggregate_rate(world, T, ms), "unit": "tokens/s", "ms_per_step": ms,
           "steps": n, "flops_per_step": fl, "block_tflops": fl / (ms / 1e3) / 1e12,
           "block_tc_frac": fl / (ms / 1e3) / 1e12 / pk["bf16_tflops"], "peak_source": f"{pk_src} bf16 burst"}
    del w, bw, x, y, ws
    torch.cuda.empty_cache()
    return out


def bench_decode_paged(args, world):
    """The 32-layer decode step of the main decode workload through the paged cache: every
    sequence's 8193 positions sit in 128-position pages spread over one pool in a random order."""
    import dataclasses

    import numpy as np
    import torch

    import llama_decoder_block_fwd_gb300 as L
    from synth import BF16, TID_KCACHE, TID_VCACHE
    from synth import configs as C
    from synth import workloads as W

    wl = C.LLAMA3_8B_DECODE
    if args.decode_layers != wl.n_layers:
        wl = dataclasses.replace(wl, n_layers=args.decode_layers, name=f"{wl.name}-L{args.decode_layers}")
    max_pos = wl.t_cache                      # the new token's position; 8193 keys
    per_seq = (max_pos + 1 + 127) // 128
    n_pages = wl.B * per_seq + 1
    perm = np.random.default_rng(wl.seed).permutation(n_pages).astype(np.int32)
    table = torch.from_numpy(perm[:wl.B * per_seq].reshape(wl.B, per_seq).copy()).cuda()
    pos = torch.full((wl.B,), max_pos, dtype=torch.int32, device="cuda")
    tensors = [W.device_layer(wl, l) for l in range(wl.n_layers)]
    layers = [L.block_weights(t) for t in tensors]
    kp = torch.empty((wl.n_layers, n_pages, 128, wl.n_kv, wl.head_dim), dtype=torch.bfloat16, device="cuda")
    vp = torch.empty_like(kp)
    for l in range(wl.n_layers):
        for tid, dst in ((TID_KCACHE, kp), (TID_VCACHE, vp)):
            dst[l].copy_(W.device_tensor(BF16, (n_pages, 128, wl.n_kv, wl.head_dim), wl.seed + l, tid, 0.0, 1.0))
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    final_g, w_lm = W.device_final(wl)
    x = W.device_x_emb(wl)
    logits = torch.empty((wl.B, wl.vocab), dtype=torch.float32, device="cuda")
    ws = torch.empty(L.llama_workspace_bytes(L.OP_STACK_DECODE_STEP, wl.dims, wl.dtype, wl.n_layers, wl.vocab,
                                             max_pos + 1), dtype=torch.uint8, device="cuda")

    def step():
        L.llama_stack_decode_step_paged(wl.dims, layers, final_g, w_lm, wl.vocab, x, kp, vp, table, pos, max_pos,
                                        logits, ws)

    step()
    L.llama_profile_read()
    L.llama_profile_enable(True)
    nprof = max(2, min(args.steps, 5))
    for _ in range(nprof):
        step()
    L.llama_profile_enable(False)
    prof = L.llama_profile_read()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(args.warmup):
        g.replay()
    barrier(world)
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        g.replay()
    e1.record(stream)
    barrier(world)
    if L.llama_get_device_status() != 0:
        raise RuntimeError("device status word set during the paged decode")
    ms = max_over_ranks(world, e0.elapsed_time(e1)) / args.steps
    pk, pk_src = peaks()
    nb = decode_bytes(wl, kv_elem_bytes=2)
    step_bytes = sum(nb.values())
    out = {"workload": wl.name + "-paged", "value": aggregate_rate(world, wl.B, ms), "unit": "tokens/s",
           "ms_per_step": ms, "bytes_per_step": step_bytes,
           "hbm_frac_step": step_bytes / (ms / 1e3) / 1e9 / pk["hbm_gbs"],
           "pages": f"{n_pages} pages of 128 positions, random order; block table [{wl.B}, {per_seq}]",
           "graph": "CUDA graph replay of one decode step"}
    attn = [k for k in prof if k.startswith("attn")]
    if attn:
        n, t = prof[attn[0]]
        per_launch = nb["kv_read"] / wl.n_layers
        ach = per_launch / (t / n / 1e3) / 1e9
        out["roofline"] = {"bound": "hbm", "kernel": attn[0], "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
                           "frac": ach / pk["hbm_gbs"], "traffic": None, "peak_source": f"{pk_src} hbm",
                           "algorithmic_bytes_per_launch": per_launch}
    del tensors, layers, kp, vp, final_g, w_lm, x, logits, ws, g, table, pos
    torch.cuda.empty_cache()
    return out


def decode_summary(d):
    """The dense decode step's headline figures, without its per-kernel record."""
    if d is None:
        return None
    r = d.get("roofline", {})
    return {"workload": d["workload"], "value": d["value"], "unit": d["unit"], "ms_per_step": d["ms_per_step"],
            "bytes_per_step": d["bytes_per_step"], "hbm_frac_step": d["hbm_frac_step"],
            "roofline": {k: r.get(k) for k in ("bound", "kernel", "achieved", "peak", "unit", "frac", "traffic")}}


# ----------------------------------------------------------------------------- oracle legs
ORACLE_SLICE = 128          # tokens per oracle step: 64 slices make up the S = 8192 sequence


def bit_reversed(n: int):
    """0..n-1 (n a power of two) in bit-reversed order: every prefix of 2^k entries is spread evenly
    over the range, so a run of oracle steps samples early and late positions alike."""
    bits = n.bit_length() - 1
    return [int(format(i, f"0{bits}b")[::-1], 2) for i in range(n)]


class OracleBlockSlices:
    """The fp64 C++ oracle on the headline workload, one Llama-3-8B block over one S = 8192 sequence,
    timed in slices of ORACLE_SLICE tokens.  Setup (not timed): draw the weights and x, and project K/V
    for all 8192 positions.  A step (timed) does the full work of one slice: it projects the slice's
    K/V again and runs the query side of every row of the slice (RMSNorm, Q, RoPE, attention over
    every key at or before the row, O + residual, RMSNorm, SwiGLU FFN + residual).  The slices of a
    run go in bit-reversed order, so the causal attention lengths of the sample match the sequence's."""

    def __init__(self):
        import oracle as O
        from synth import configs as C
        from synth import workloads as W
        self.O = O
        self.wl = wl = C.LLAMA3_8B_PREFILL
        self.hw = O.BlockWeights(**W.host_layer(wl))
        self.x = W.host_x(wl, 0)[None]
        self.dims = O.Dims(1, wl.S, wl.d_model, wl.n_q, wl.n_kv, wl.head_dim, wl.d_ff, wl.theta_base, wl.eps)
        self.k, self.v = O.project_kv(self.x, self.hw, self.dims)
        self.order = bit_reversed(wl.S // ORACLE_SLICE)
        self.threads = O.threads()

    def step(self, j: int) -> float:
        """Seconds for slice order[j mod 64]."""
        import dataclasses

        import numpy as np
        O, n = self.O, ORACLE_SLICE
        s0 = self.order[j % len(self.order)] * n
        t0 = time.perf_counter()
        O.project_kv(self.x[:, s0:s0 + n], self.hw, dataclasses.replace(self.dims, S=n), pos0=s0)
        O.block_rows(self.x, self.hw, self.dims, self.k, self.v, np.arange(s0, s0 + n))
        return time.perf_counter() - t0

    def sample(self, steps: int, seconds: float) -> str:
        return (f"{self.wl.name}: K/V of all {self.wl.S} positions projected before the clock; {steps} timed "
                f"steps of one {ORACLE_SLICE}-token slice each (its K/V projection and the query side of all "
                f"its rows, attending to every earlier key), slices in bit-reversed order over the sequence; "
                f"fp64 C++ oracle, {self.threads} OpenMP threads, {seconds:.1f} s")


def prefill_config(wl, world: int, step_flops: float) -> dict:
    """The headline workload's config record (the same on both arms of the bench)."""
    return {"workload": wl.name, "B": wl.B, "S": wl.S, "d_model": wl.d_model, "n_q": wl.n_q,
            "n_kv": wl.n_kv, "head_dim": wl.head_dim, "d_ff": wl.d_ff, "theta_base": wl.theta_base,
            "eps": wl.eps, "global_batch": world * wl.B, "seq_len": wl.S, "parallelism": f"replicas{world}",
            "l2": "inputs larger than L2 (436 MB of weights + 64 MB activations per step)",
            "flops_per_step": step_flops}


def cpu_baseline(n_steps: int = 8) -> dict:
    """The oracle on n_steps slices of the headline workload (~10-30 s on the host cores)."""
    o = OracleBlockSlices()
    total = sum(o.step(j) for j in range(n_steps))
    return {"value": n_steps * ORACLE_SLICE / total, "unit": "tokens/s", "cores": o.threads, "kind": "oracle",
            "sample": o.sample(n_steps, total)}


def run_reference(args, world):
    from synth import configs as C
    wl = C.LLAMA3_8B_PREFILL
    o = OracleBlockSlices()
    for j in range(args.warmup):
        o.step(args.steps + j)          # warm-up slices lie outside the timed steps' slices
    times = [o.step(j) for j in range(args.steps)]
    total = sum(times)
    ms = 1e3 * total / args.steps
    val = ORACLE_SLICE / (ms / 1e3)
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,0.02) weights, N(0,1) inputs)",
        "config": prefill_config(wl, world, sum(prefill_flops(wl).values())),
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": o.threads, "kind": "oracle",
                         "sample": o.sample(args.steps, total)},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-mha", action="store_true", help="skip the LLaMA-7B MHA block prefill")
    ap.add_argument("--no-kv8", action="store_true", help="skip the decode step over an 8-bit KV cache")
    ap.add_argument("--no-chunked", action="store_true", help="skip the chunked-prefill line")
    ap.add_argument("--no-paged", action="store_true", help="skip the paged-cache decode line")
    ap.add_argument("--no-long", action="store_true", help="skip the 32K-context prefill and decode lines")
    ap.add_argument("--no-rmsnorm", action="store_true", help="skip the standalone RMSNorm line")
    ap.add_argument("--rmsnorm-rows", type=int, default=8192, help="rows of the standalone RMSNorm line")
    ap.add_argument("--only", choices=["prefill", "decode", "decode_kv8", "rmsnorm", "sample"],
                    help="run this one line alone and print its record (for profiler captures)")
    ap.add_argument("--prefill-seq", type=int, default=8192, help="tokens of the prefill workload (default 8192)")
    ap.add_argument("--decode-layers", type=int, default=32, help="layers of the decode stack (default 32)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        if int(os.environ.get("RANK", "0")) == 0:
            run_reference(args, world)
        return

    world, rank, local = dist_setup()
    if args.only:   # a profiling aid: one line alone
        rec = {"prefill": lambda: bench_prefill(args, world, rank),
               "decode": lambda: bench_decode(args, world, rank),
               "decode_kv8": lambda: bench_decode(args, world, rank, kv8=True),
               "rmsnorm": lambda: bench_rmsnorm(args, world),
               "sample": lambda: bench_sample(args, world)}[args.only]()
        if rank == 0:
            print(json.dumps({args.only: rec}), flush=True)
        return
    pre = bench_prefill(args, world, rank)
    mha = None if args.no_mha else bench_mha_prefill(args, world)
    dec = None if args.no_decode else bench_decode(args, world, rank)
    dec8 = None if (args.no_decode or args.no_kv8) else bench_decode(args, world, rank, kv8=True)
    smp = None if args.no_decode else bench_sample(args, world)
    chk = None if args.no_chunked else bench_chunked_prefill(args, world)
    pgd = None if (args.no_decode or args.no_paged) else bench_decode_paged(args, world)
    lpre = None if args.no_long else bench_prefill_long(args, world)
    ldec = None if (args.no_decode or args.no_long) else bench_decode(args, world, rank, seqs=16, cached=32768)
    rms = None if args.no_rmsnorm else bench_rmsnorm(args, world)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline()
    if rank == 0:
        line = {
            "metric": METRIC, "value": pre["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": pre["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,0.02) weights, N(0,1) inputs)",
            "config": pre["config"], "roofline": pre["roofline"], "cpu_baseline": cpu, "e2e": pre["e2e"],
            "gpu_launches": pre["gpu_launches"], "clocks": pre["clocks"], "block_tc_frac": pre["block_tc_frac"],
            "block_tflops": pre["block_tflops"], "kernels": pre["kernels"], "prefill_sustained": pre["sustained"],
            "decode_detail": dec, "mha_prefill": mha, "decode_kv8": dec8, "sample": smp, "chunked_prefill": chk,
            "decode_paged": pgd, "prefill_32k": lpre, "decode_32k": ldec, "rmsnorm": rms,
            # last, so that a reader of the line's tail sees it: the 32-layer B64 x 8192 dense decode step
            "decode": decode_summary(dec),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
