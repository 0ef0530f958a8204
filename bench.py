"""Benchmark: elu+1 kernelized linear attention on GB300.

Headline step: one causal chunkwise forward (la_forward_causal) over the
B=8, H=16, N=8192, d=dv=128 bf16 workload (tokens = B*N positions, all heads).
Each extra mode (non-causal B4 H8 N4096 d64, long causal B1 H32 N131072 d64,
recurrent decode B256 H32 d128, gradients of the causal form at B8 H16 N8192
d128, and the per-head decay variants: causal B8 H16 N8192 d128 and decode
B256 H32 d128) is timed the same way and reported under "modes" with its own
roofline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same per-GPU workload (weak
scaling, no data-path collective); timing is the max over ranks.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from linear_rnn_sequence_gb300.workloads import (WORKLOADS, Workload, head_decays,  # noqa: E402
                                                 make_backward_inputs, make_gated_inputs,
                                                 make_qkv)

METRIC = "causal linear-attn tokens/s & TFLOP/s on 1 GB300, % roofline; decode tokens/s"
HEADLINE = "causal_bf16_b8h16n8192d128"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------
# algorithmic counts (per token-head; decode: per head-step)
# ----------------------------------------------------------------------------
def esize(dt):
    return 2 if dt == torch.bfloat16 else 4


def alg_flops_per_token_head(d, dv):
    # state update 2*d*dv, query 2*d*dv, z update d, phi(q).z 2d, divide dv
    return 4 * d * dv + 3 * d + dv


def alg_bytes_per_token_head(w: Workload):
    """Algorithmic bytes: q, k, v read and y written once, all at the input dtype."""
    return (2 * w.d + 2 * w.dv) * esize(w.dtype)


def moved_bytes_per_token_head(w: Workload):
    """The same with y written as float32, as the library writes it."""
    return (2 * w.d + w.dv) * esize(w.dtype) + w.dv * 4


def bwd_flops_per_token_head(d, dv):
    # forward direction: S update 2*d*dv, S g 2*d*dv; reverse: Sh update
    # 2*d*dv, Sh v 2*d*dv, Sh^T phi(k) 2*d*dv; plus den, e, z e, zh terms
    return 10 * d * dv + 8 * d + 4 * dv


def bwd_bytes_per_token_head(w: Workload):
    # q, k, v read; dy (fp32) read; dq, dk, dv (fp32) written
    return (2 * w.d + w.dv) * esize(w.dtype) + w.dv * 4 + (2 * w.d + w.dv) * 4


# fp32 FMA peak of the CUDA cores: 152 SMs x 128 FP32 lanes x 2 FLOP x 2.07 GHz
ALU_FP32_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def decay_flops_per_token_head(d, dv):
    # the recurrent definition: decay of S (d*dv) and z (d), update 2*d*dv + d,
    # query 2*d*dv + 2d + dv
    return 5 * d * dv + 4 * d + dv


def decode_bytes_per_head_step(w: Workload):
    """fp32 S and z read and written; q, k, v read and y written at the input dtype."""
    return 2 * (w.d * w.dv + w.d) * 4 + (2 * w.d + 2 * w.dv) * esize(w.dtype)


def decode_moved_bytes_per_head_step(w: Workload):
    """The same with y written as float32."""
    return 2 * (w.d * w.dv + w.d) * 4 + (2 * w.d + w.dv) * esize(w.dtype) + w.dv * 4


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------
# distributed plumbing
# ----------------------------------------------------------------------------
def dist_setup(gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The slowest rank's figure, on every rank (NCCL on the GPUs, gloo on CPU)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, ms_per_step: float) -> float:
    """Units all ranks processed per second, timed by the slowest rank.

    Every rank runs the same per-GPU workload (weak scaling, replicas), so the
    job processes world * units_per_rank units per step."""
    return world * units_per_rank / (ms_per_step * 1e-3)


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, local_rank):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        idx = str(local_rank)
        if vis:
            parts = [p.strip() for p in vis.split(",")]
            if local_rank < len(parts) and parts[local_rank].isdigit():
                idx = parts[local_rank]
        self.idx = idx
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.idx, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not getattr(self, "out", ""):
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------
# timing helpers
# ----------------------------------------------------------------------------
def flush_l2(buf):
    buf.zero_()


def time_steps(fn, steps, warmup, world, flush=None, min_warm_s=0.0):
    """Run `warmup` untimed steps, then exactly `steps` timed steps.

    Warm-up continues (untimed) until at least `min_warm_s` seconds have
    passed, so that clock samples taken alongside see the GPU under load.
    Returns (total_ms (max over ranks), per-step kernel ms list from events on
    the launching stream).  If `flush` is given it runs between timed steps,
    outside the per-step event pairs.
    """
    stream = torch.cuda.current_stream()
    t_warm = time.perf_counter()
    for _ in range(warmup):   # the warm-up repeats the timed loop's pattern, flush included
        if flush is not None:
            flush()
        fn()
    torch.cuda.synchronize()
    while time.perf_counter() - t_warm < min_warm_s:
        for _ in range(8):
            fn()
        torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(steps):
        if flush is not None:
            flush()
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    per = [a.elapsed_time(b) for a, b in ev]
    total = sum(per) if flush is not None else t_start.elapsed_time(t_end)
    return max_over_ranks(total, world), per


BYTES_BASIS = "q, k, v read and y written once at the input dtype (decode: plus fp32 S, z read and written)"


def roofline(bytes_per_launch, flops_per_launch, launch_ms, peaks, peak_kind, traffic=None,
             moved_bytes=None):
    """Achieved rate and fraction of the measured peak for one launch.

    ``frac`` is on the algorithmic bytes (BYTES_BASIS).  ``fp32_y`` repeats
    the bytes figure with y counted as float32, the bytes the kernels move."""
    t = launch_ms * 1e-3
    gbs = bytes_per_launch / t / 1e9
    tflops = flops_per_launch / t / 1e12
    t_bytes = bytes_per_launch / (peaks["hbm_gbs"] * 1e9)
    t_flops = flops_per_launch / (peaks["bf16_tflops"] * 1e12)
    if t_bytes >= t_flops:
        r = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
             "frac": gbs / peaks["hbm_gbs"]}
    else:
        r = {"bound": "tensor", "achieved": tflops, "peak": peaks["bf16_tflops"],
             "unit": "TFLOP/s", "frac": tflops / peaks["bf16_tflops"]}
    r["traffic"] = traffic
    r["peak_source"] = peak_kind
    r["roof_fraction"] = max(t_bytes, t_flops) / t  # slower of the two roofs / measured time
    r["bytes_basis"] = BYTES_BASIS
    r["bytes_per_launch"] = bytes_per_launch
    if moved_bytes is not None:
        gbs = moved_bytes / t / 1e9
        r["fp32_y"] = {"bytes_per_launch": moved_bytes, "achieved_gbs": gbs,
                       "frac": gbs / peaks["hbm_gbs"]}
    return r


# ----------------------------------------------------------------------------
# CPU baseline: the fp64 oracle as it stands, on a bounded sample
# ----------------------------------------------------------------------------
def cpu_baseline(w: Workload, budget_s=12.0, budget_1t_s=4.0):
    """The oracle on the host cores (all of them, then one thread), in tokens/s
    of the workload: B*N positions across all H heads."""
    import oracle
    cores = oracle.default_threads()
    sample = w.with_(B=1)
    q, k, v = make_qkv(sample)
    done_tokens, t0 = 0, time.perf_counter()
    reps = 0
    while True:
        oracle.causal_recurrent(q, k, v, eps=w.eps, nthreads=cores)
        reps += 1
        done_tokens += sample.N  # one batch row: N positions with all H heads
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    # one thread: whole heads of the same row, one after another; a position
    # needs all H heads, so the rate is N / (H x seconds per head)
    heads, t1 = 0, time.perf_counter()
    while True:
        h = heads % w.H
        oracle.causal_recurrent(q[:, h:h + 1], k[:, h:h + 1], v[:, h:h + 1], eps=w.eps, nthreads=1)
        heads += 1
        if time.perf_counter() - t1 >= budget_1t_s:
            break
    el1 = time.perf_counter() - t1
    return {"value": done_tokens / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{reps} x (B=1, H={w.H}, N={w.N}, d={w.d}, dv={w.dv}) recurrent fp64, "
                      f"{el:.1f} s; one thread: {heads} heads of that row, {el1:.1f} s",
            "value_1thread": sample.N / (w.H * el1 / heads)}


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------
def run_ours(args, world, rank, local):
    from linear_rnn_sequence_gb300 import linattn as la
    dev = torch.device("cuda", local)
    peaks, peak_kind = load_peaks()
    w = WORKLOADS[HEADLINE]
    q, k, v = make_qkv(w, device=dev, gen_device=dev)
    y = torch.empty(w.B, w.H, w.N, w.dv, device=dev)
    need = la.causal_workspace_bytes(w.B, w.H, w.N, w.d, w.dv, w.dtype)
    ws = la.alloc_workspace(need, dev)

    def step():
        la.forward_causal(q, k, v, eps=w.eps, out=y, workspace=ws)

    # clocks: sampled every 50 ms from the start of the (load-keeping) warm-up
    # through the timed steps
    with ClockSampler(local) as clk:
        total_ms, per = time_steps(step, args.steps, args.warmup, world, min_warm_s=0.6)
    clocks = clk.summary()
    T = w.B * w.H * w.N
    tokens = w.B * w.N
    ms_per_step = total_ms / args.steps
    value = whole_job_rate(tokens, world, ms_per_step)
    launch_ms = sum(per) / len(per)
    bytes_launch = T * alg_bytes_per_token_head(w)
    flops_launch = T * alg_flops_per_token_head(w.d, w.dv)
    traffic = load_traffic(HEADLINE)
    roof = roofline(bytes_launch, flops_launch, launch_ms, peaks, peak_kind, traffic,
                    moved_bytes=T * moved_bytes_per_token_head(w))
    status = la.workspace_status(ws)

    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": path_dtype(w), "data": "synthetic (seeded iid N(0,1)/sqrt(d), bf16)",
        "config": {"workload": HEADLINE, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "dv": w.dv,
                   "input_dtype": "bf16", "output_dtype": "f32", "eps": w.eps,
                   "l2": "inputs larger than L2 (1.07 GB of q,k,v per step)",
                   "parallelism": f"replica x{world}"},
        "tflops": world * flops_launch / (ms_per_step * 1e-3) / 1e12,
        "roofline": roof,
        "gpu_launches": args.steps * launches_per_call("causal", w),
        "clocks": clocks,
        "run_status": la.status_string(status),
    }
    del q, k, v, y
    torch.cuda.empty_cache()
    if not args.no_e2e:
        out["e2e"] = e2e_causal(w, dev, world, args)
    if not args.no_modes:
        out["modes"] = run_modes(args, world, dev, peaks, peak_kind)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w)
    return out


def path_dtype(w):
    from linear_rnn_sequence_gb300 import linattn as la
    tc = la.causal_workspace_bytes(w.B, w.H, w.N, w.d, w.dv, w.dtype) > 0
    return "bf16" if (tc and w.dtype == torch.bfloat16) else "f32"


def launches_per_call(mode, w):
    """Kernels of ours that one call launches (the launch list under ncu agrees).

    A causal call launches one kernel, or three (segment states, their prefix
    scan, the chunk kernel) when the workspace holds segment states, i.e. when
    it is larger than its 256-byte header.
    """
    from linear_rnn_sequence_gb300 import linattn as la
    if mode == "causal":
        return 3 if la.causal_workspace_bytes(w.B, w.H, w.N, w.d, w.dv, w.dtype) > 256 else 1
    tc = w.dtype == torch.bfloat16 and w.d in (64, 128) and w.dv in (64, 128)
    if mode == "noncausal":
        # tensor-core path (bf16, d and dv in {64, 128}): one fused kernel
        # (partial states, their per-head sum, the queries); otherwise two
        # CUDA-core kernels
        return 1 if tc else 2
    if mode == "causal_decay":
        # tensor-core kernel for the heads it takes (preceded by the segment
        # states and their prefix scan when the sequence is split), then the
        # CUDA-core kernel for the rest (its CTAs for the first kind return)
        if not tc:
            return 1
        split = la.causal_workspace_bytes(w.B, w.H, w.N, w.d, w.dv, w.dtype) > 256
        return 4 if split else 2
    return 1


def load_traffic(name):
    """DRAM bytes per launch of the dominant kernel, from a committed ncu summary.

    The entry lists the sources the kernel was built from and their sha256 at
    capture time; once any of them has changed the figure no longer describes
    the kernel that runs, and null is returned.
    """
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            e = json.load(f)["workloads"].get(name)
        if not e:
            return None
        h = hashlib.sha256()
        for src in e["sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        return int(e["bytes"]) if h.hexdigest() == e["sha256"] else None
    except Exception:
        return None


def e2e_causal(w, dev, world, args):
    """Same metric end to end through the C ABI on HOST buffers
    (la_forward_causal_host): every step uploads q, k, v from page-locked host
    memory, runs the forward and downloads y, with the copies of one head group
    overlapping the kernels and copies of the others.  The call returns when y
    is in host memory, so the timed region covers all of it."""
    from linear_rnn_sequence_gb300 import linattn as la
    qh, kh, vh = (t.pin_memory() for t in make_qkv(w.with_(B=1), device="cpu"))
    # one batch row drawn, replicated to B rows (keeps the draw fast)
    qh = qh.expand(w.B, -1, -1, -1).contiguous().pin_memory()
    kh = kh.expand(w.B, -1, -1, -1).contiguous().pin_memory()
    vh = vh.expand(w.B, -1, -1, -1).contiguous().pin_memory()
    yh = torch.empty(w.B, w.H, w.N, w.dv, dtype=torch.float32).pin_memory()
    buf = la.alloc_workspace(la.causal_host_buffer_bytes(w.B, w.H, w.N, w.d, w.dv, w.dtype), dev)

    def step():
        la.forward_causal_host(qh, kh, vh, eps=w.eps, out=yh, dev_buf=buf, device=dev)

    steps = max(3, min(args.steps, 10))
    total_ms, _ = time_steps(step, steps, 2, world)
    ms = total_ms / steps
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
    d2h = yh.numel() * yh.element_size()
    return {"value": world * w.B * w.N / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "api": "la_forward_causal_host (pinned host buffers, copies overlapped with kernels)"}


def run_modes(args, world, dev, peaks, peak_kind):
    from linear_rnn_sequence_gb300 import linattn as la
    modes = {}
    flush_buf = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    steps = max(3, min(args.steps, 20))

    # non-causal: inputs fit in L2, so flush L2 between timed launches
    w = WORKLOADS["noncausal_bf16_b4h8n4096d64"]
    q, k, v = make_qkv(w, device=dev, gen_device=dev)
    y = torch.empty(w.B, w.H, w.N, w.dv, device=dev)
    ws = la.alloc_workspace(la.noncausal_workspace_bytes(w.B, w.H, w.N, w.d, w.dv), dev)
    total, per = time_steps(lambda: la.forward_noncausal(q, k, v, out=y, workspace=ws), steps,
                            args.warmup, world, flush=lambda: flush_l2(flush_buf))
    T = w.BH * w.N
    ms = sum(per) / len(per)
    modes[w.name] = {"tokens_per_s": world * w.B * w.N / (ms * 1e-3), "ms_per_call": ms,
                     "l2": "flushed between launches (256 MB write)",
                     "roofline": roofline(T * alg_bytes_per_token_head(w),
                                          T * alg_flops_per_token_head(w.d, w.dv), ms, peaks,
                                          peak_kind, load_traffic(w.name),
                                          moved_bytes=T * moved_bytes_per_token_head(w))}
    del q, k, v, y, ws

    # long causal
    w = WORKLOADS["causal_bf16_b1h32n131072d64"]
    q, k, v = make_qkv(w, device=dev, gen_device=dev)
    y = torch.empty(w.B, w.H, w.N, w.dv, device=dev)
    ws = la.alloc_workspace(la.causal_workspace_bytes(w.B, w.H, w.N, w.d, w.dv, w.dtype), dev)
    total, per = time_steps(lambda: la.forward_causal(q, k, v, out=y, workspace=ws), steps,
                            args.warmup, world)
    T = w.BH * w.N
    ms = sum(per) / len(per)
    modes[w.name] = {"tokens_per_s": world * w.B * w.N / (ms * 1e-3), "ms_per_call": ms,
                     "l2": "inputs larger than L2",
                     "roofline": roofline(T * alg_bytes_per_token_head(w),
                                          T * alg_flops_per_token_head(w.d, w.dv), ms, peaks,
                                          peak_kind, load_traffic(w.name),
                                          moved_bytes=T * moved_bytes_per_token_head(w))}
    del q, k, v, y, ws
    torch.cuda.empty_cache()

    # decode: state from a 1024-token prefill, then timed steps (state > L2)
    w = WORKLOADS["decode_bf16_b256h32d128"]
    q, k, v = make_qkv(w, device=dev, gen_device=dev)
    _, S, z = la.forward_causal(q, k, v, return_state=True)
    del q, k, v
    torch.cuda.empty_cache()
    # the workload's 4096 steps, each on one of 256 pre-drawn (q, k, v) sets in
    # turn (drawing all 4096 would take 25 GB); the state evolves step by step
    nsets, nsteps = 256, w.steps
    g = torch.Generator(device=dev).manual_seed(w.seed + 1)
    sc = torch.tensor(w.step_scale, device=dev)
    qs = (torch.randn(nsets, w.B, w.H, w.d, generator=g, device=dev) * sc).to(w.dtype)
    ks = (torch.randn(nsets, w.B, w.H, w.d, generator=g, device=dev) * sc).to(w.dtype)
    vs = (torch.randn(nsets, w.B, w.H, w.dv, generator=g, device=dev) * sc).to(w.dtype)
    yd = torch.empty(w.B, w.H, w.dv, device=dev)
    it = [0]

    def dstep():
        i = it[0] % nsets
        it[0] += 1
        la.decode_step(qs[i], ks[i], vs[i], S, z, eps=w.eps, out=yd)

    total, per = time_steps(dstep, nsteps, args.warmup, world)
    ms = total / nsteps
    heads = w.BH
    roof = roofline(heads * decode_bytes_per_head_step(w), heads * alg_flops_per_token_head(w.d, w.dv),
                    sum(per) / len(per), peaks, peak_kind, load_traffic(w.name),
                    moved_bytes=heads * decode_moved_bytes_per_head_step(w))
    # per step over the whole run, launch gaps included (the per-launch figure
    # above can read a little high: part of a step's write-back is still in L2)
    roof["frac_per_step"] = heads * decode_bytes_per_head_step(w) / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"]
    modes[w.name] = {"tokens_per_s": world * w.B / (ms * 1e-3), "ms_per_step": ms,
                     "steps_timed": nsteps, "l2": "state (512 MB) larger than L2",
                     "roofline": roof}
    del qs, ks, vs, S, z
    torch.cuda.empty_cache()

    # gradients of the causal form (CUDA cores, fp32): inputs larger than L2
    w = WORKLOADS["causal_backward_bf16_b8h16n8192d128"]
    q, k, v, dy = make_backward_inputs(w, device=dev, gen_device=dev)
    outs = (torch.empty(w.B, w.H, w.N, w.d, device=dev), torch.empty(w.B, w.H, w.N, w.d, device=dev),
            torch.empty(w.B, w.H, w.N, w.dv, device=dev))
    ws = la.alloc_workspace(la.causal_backward_workspace_bytes(w.B, w.H, w.N, w.d, w.dv, w.dtype),
                            dev)
    total, per = time_steps(lambda: la.backward_causal(q, k, v, dy, eps=w.eps, out=outs,
                                                       workspace=ws),
                            max(3, min(args.steps, 10)), args.warmup, world)
    T = w.BH * w.N
    ms = sum(per) / len(per)
    alg_flops, alg_bytes = T * bwd_flops_per_token_head(w.d, w.dv), T * bwd_bytes_per_token_head(w)
    tflops = alg_flops / (ms * 1e-3) / 1e12
    modes[w.name] = {"tokens_per_s": world * w.B * w.N / (ms * 1e-3), "ms_per_call": ms,
                     "l2": "inputs larger than L2",
                     "roofline": {"bound": "alu", "achieved": tflops, "peak": ALU_FP32_TFLOPS,
                                  "unit": "TFLOP/s", "frac": tflops / ALU_FP32_TFLOPS,
                                  "traffic": load_traffic("causal_backward_bf16_b8h16n8192d128"),
                                  "peak_source": "fp32 FMA: 152 SMs x 128 lanes x 2 FLOP x 2.07 GHz",
                                  "hbm_roof_fraction": alg_bytes / (peaks["hbm_gbs"] * 1e9) / (ms * 1e-3)}}
    # the same gradients for the decayed forward (per-head gamma)
    gam = head_decays(w.H).to(dev)
    total, per = time_steps(lambda: la.backward_causal(q, k, v, dy, eps=w.eps, out=outs,
                                                       workspace=ws, gamma=gam),
                            max(3, min(args.steps, 10)), args.warmup, world)
    ms = sum(per) / len(per)
    # the decayed recurrence adds one multiply per state element in each
    # direction: 12 d dv instead of 10 d dv
    alg_flops = T * (bwd_flops_per_token_head(w.d, w.dv) + 2 * w.d * w.dv)
    tflops = alg_flops / (ms * 1e-3) / 1e12
    modes["causal_backward_decay_bf16_b8h16n8192d128"] = {
        "tokens_per_s": world * w.B * w.N / (ms * 1e-3), "ms_per_call": ms,
        "l2": "inputs larger than L2",
        "roofline": {"bound": "alu", "achieved": tflops, "peak": ALU_FP32_TFLOPS,
                     "unit": "TFLOP/s", "frac": tflops / ALU_FP32_TFLOPS,
                     "traffic": load_traffic("causal_backward_decay_bf16_b8h16n8192d128"),
                     "peak_source": "fp32 FMA: 152 SMs x 128 lanes x 2 FLOP x 2.07 GHz",
                     "hbm_roof_fraction": alg_bytes / (peaks["hbm_gbs"] * 1e9) / (ms * 1e-3)}}
    del q, k, v, dy, outs, ws
    torch.cuda.empty_cache()

    # gated causal (one gate per token and head, all in [3/4, 1): every head on
    # the tensor cores, after the per-block tables of gate products)
    w = WORKLOADS["causal_gated_bf16_b8h16n8192d128"]
    q, k, v, gate = make_gated_inputs(w, device=dev, gen_device=dev)
    y = torch.empty(w.B, w.H, w.N, w.dv, device=dev)
    ws = la.alloc_workspace(la.causal_gated_workspace_bytes(w.B, w.H, w.N, w.d, w.dv, w.dtype), dev)
    total, per = time_steps(lambda: la.forward_causal_gated(q, k, v, gate=gate, eps=w.eps, out=y,
                                                            workspace=ws),
                            steps, args.warmup, world)
    T = w.BH * w.N
    ms = sum(per) / len(per)
    gate_bytes = T * 4   # the fp32 gates, read once
    modes[w.name] = {"tokens_per_s": world * w.B * w.N / (ms * 1e-3), "ms_per_call": ms,
                     "l2": "inputs larger than L2", "kernels_per_call": 3,
                     "roofline": roofline(T * alg_bytes_per_token_head(w) + gate_bytes,
                                          T * decay_flops_per_token_head(w.d, w.dv), ms, peaks,
                                          peak_kind, load_traffic(w.name),
                                          moved_bytes=T * moved_bytes_per_token_head(w) + gate_bytes)}
    del q, k, v, gate, y, ws
    torch.cuda.empty_cache()

    # causal with a per-head decay (every head of this workload has
    # gamma >= 2^-1/2, so the tensor-core kernel computes all of them; the
    # CUDA-core pass that follows only returns)
    w = WORKLOADS["causal_decay_bf16_b8h16n8192d128"]
    q, k, v = make_qkv(w, device=dev, gen_device=dev)
    gam = head_decays(w.H).to(dev)
    y = torch.empty(w.B, w.H, w.N, w.dv, device=dev)
    ws = la.alloc_workspace(la.causal_workspace_bytes(w.B, w.H, w.N, w.d, w.dv, w.dtype), dev)
    total, per = time_steps(lambda: la.forward_causal_decay(q, k, v, gam, eps=w.eps, out=y,
                                                            workspace=ws),
                            max(3, min(args.steps, 10)), args.warmup, world)
    T = w.BH * w.N
    ms = sum(per) / len(per)
    modes[w.name] = {"tokens_per_s": world * w.B * w.N / (ms * 1e-3), "ms_per_call": ms,
                     "l2": "inputs larger than L2",
                     "kernels_per_call": launches_per_call("causal_decay", w),
                     "roofline": roofline(T * alg_bytes_per_token_head(w),
                                          T * decay_flops_per_token_head(w.d, w.dv), ms, peaks,
                                          peak_kind, load_traffic(w.name),
                                          moved_bytes=T * moved_bytes_per_token_head(w))}
    del q, k, v, y, ws
    torch.cuda.empty_cache()

    # long-context causal with a per-head decay: few heads, so the sequence is
    # split (decayed segment states, their decayed prefix scan, chunk kernel)
    w = WORKLOADS["causal_decay_bf16_b1h32n131072d64"]
    q, k, v = make_qkv(w, device=dev, gen_device=dev)
    gam = head_decays(w.H).to(dev)
    y = torch.empty(w.B, w.H, w.N, w.dv, device=dev)
    ws = la.alloc_workspace(la.causal_workspace_bytes(w.B, w.H, w.N, w.d, w.dv, w.dtype), dev)
    total, per = time_steps(lambda: la.forward_causal_decay(q, k, v, gam, eps=w.eps, out=y,
                                                            workspace=ws),
                            steps, args.warmup, world)
    T = w.BH * w.N
    ms = sum(per) / len(per)
    modes[w.name] = {"tokens_per_s": world * w.B * w.N / (ms * 1e-3), "ms_per_call": ms,
                     "l2": "inputs larger than L2",
                     "kernels_per_call": launches_per_call("causal_decay", w),
                     "roofline": roofline(T * alg_bytes_per_token_head(w),
                                          T * decay_flops_per_token_head(w.d, w.dv), ms, peaks,
                                          peak_kind, load_traffic(w.name),
                                          moved_bytes=T * moved_bytes_per_token_head(w))}
    del q, k, v, y, ws
    torch.cuda.empty_cache()

    # decode with a per-head decay: state from a decayed 1024-token prefill
    w = WORKLOADS["decode_decay_bf16_b256h32d128"]
    gam = head_decays(w.H).to(dev)
    q, k, v = make_qkv(w, device=dev, gen_device=dev)
    _, S, z = la.forward_causal_decay(q, k, v, gam, return_state=True)
    del q, k, v
    torch.cuda.empty_cache()
    g = torch.Generator(device=dev).manual_seed(w.seed + 1)
    sc = torch.tensor(w.step_scale, device=dev)
    qs = (torch.randn(nsets, w.B, w.H, w.d, generator=g, device=dev) * sc).to(w.dtype)
    ks = (torch.randn(nsets, w.B, w.H, w.d, generator=g, device=dev) * sc).to(w.dtype)
    vs = (torch.randn(nsets, w.B, w.H, w.dv, generator=g, device=dev) * sc).to(w.dtype)
    it[0] = 0

    def ddstep():
        i = it[0] % nsets
        it[0] += 1
        la.decode_step_decay(qs[i], ks[i], vs[i], S, z, gam, eps=w.eps, out=yd)

    nsteps = w.steps
    total, per = time_steps(ddstep, nsteps, args.warmup, world)
    ms = total / nsteps
    roof = roofline(w.BH * decode_bytes_per_head_step(w), w.BH * decay_flops_per_token_head(w.d, w.dv),
                    sum(per) / len(per), peaks, peak_kind, load_traffic(w.name),
                    moved_bytes=w.BH * decode_moved_bytes_per_head_step(w))
    roof["frac_per_step"] = w.BH * decode_bytes_per_head_step(w) / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"]
    modes[w.name] = {"tokens_per_s": world * w.B / (ms * 1e-3), "ms_per_step": ms,
                     "steps_timed": nsteps, "l2": "state (512 MB) larger than L2",
                     "roofline": roof}
    del qs, ks, vs, S, z
    torch.cuda.empty_cache()
    return modes


# ----------------------------------------------------------------------------
# reference arm: the oracle, as it stands, on the host cores
# ----------------------------------------------------------------------------
def run_reference(args, world, rank):
    if rank != 0:
        return None
    import oracle
    w = WORKLOADS[HEADLINE]
    cores = oracle.default_threads()
    sample = w.with_(B=1, N=1024)   # one batch row, first 1024 positions, all heads
    q, k, v = make_qkv(sample)
    for _ in range(args.warmup):
        oracle.causal_recurrent(q[:, :, :64], k[:, :, :64], v[:, :, :64], nthreads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.causal_recurrent(q, k, v, eps=w.eps, nthreads=cores)
    el = time.perf_counter() - t0
    value = args.steps * sample.N / el
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": HEADLINE, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "dv": w.dv},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"each step: B=1, H={w.H}, N={sample.N}, d={w.d} "
                                       f"recurrent fp64"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def profile_case(args):
    """A few launches of one kernel on one workload, for ncu captures.

    --profile-case causal|long|noncausal|decode|backward|backward_decay|causal_decay|
    long_decay|decode_decay|gated picks the workload (B8 H16 N8192 d128 / B1 H32
    N131072 d64 / B4 H8 N4096 d64 / B256 H32 d128 decode / gradients at B8 H16 N8192
    d128, without and with the per-head decays / the decay variants of the causal,
    long and decode workloads / the gated causal form at B8 H16 N8192 d128);
    --batch overrides B for a smaller capture.
    """
    from linear_rnn_sequence_gb300 import linattn as la
    names = {"causal": HEADLINE, "long": "causal_bf16_b1h32n131072d64",
             "noncausal": "noncausal_bf16_b4h8n4096d64", "decode": "decode_bf16_b256h32d128",
             "backward": "causal_backward_bf16_b8h16n8192d128",
             "backward_decay": "causal_backward_bf16_b8h16n8192d128",
             "causal_decay": "causal_decay_bf16_b8h16n8192d128",
             "long_decay": "causal_decay_bf16_b1h32n131072d64",
             "decode_decay": "decode_decay_bf16_b256h32d128",
             "gated": "causal_gated_bf16_b8h16n8192d128"}
    w = WORKLOADS[names[args.profile_case]]
    if args.batch:
        w = w.with_(B=args.batch)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if w.mode in ("decode", "decode_decay"):
        g = torch.Generator(device=dev).manual_seed(w.seed + 1)
        sc = torch.tensor(w.step_scale, device=dev)
        S = torch.randn(w.B, w.H, w.d, w.dv, generator=g, device=dev)
        z = torch.rand(w.B, w.H, w.d, generator=g, device=dev) * 1000 + 1
        q, k = ((torch.randn(w.B, w.H, w.d, generator=g, device=dev) * sc).to(w.dtype) for _ in range(2))
        v = (torch.randn(w.B, w.H, w.dv, generator=g, device=dev) * sc).to(w.dtype)
        y = torch.empty(w.B, w.H, w.dv, device=dev)
        if w.mode == "decode":
            fn = lambda: la.decode_step(q, k, v, S, z, eps=w.eps, out=y)
        else:
            gam = head_decays(w.H).to(dev)
            fn = lambda: la.decode_step_decay(q, k, v, S, z, gam, eps=w.eps, out=y)
    elif args.profile_case == "gated":
        q, k, v, gate = make_gated_inputs(w, device=dev, gen_device=dev)
        y = torch.empty(w.B, w.H, w.N, w.dv, device=dev)
        fn = lambda: la.forward_causal_gated(q, k, v, gate=gate, eps=w.eps, out=y)
    elif w.mode == "causal_decay":
        q, k, v = make_qkv(w, device=dev, gen_device=dev)
        y = torch.empty(w.B, w.H, w.N, w.dv, device=dev)
        gam = head_decays(w.H).to(dev)
        ws = la.alloc_workspace(la.causal_workspace_bytes(w.B, w.H, w.N, w.d, w.dv, w.dtype), dev)
        fn = lambda: la.forward_causal_decay(q, k, v, gam, eps=w.eps, out=y, workspace=ws)
    elif w.mode == "backward":
        q, k, v, dy = make_backward_inputs(w, device=dev, gen_device=dev)
        outs = (torch.empty(w.B, w.H, w.N, w.d, device=dev),
                torch.empty(w.B, w.H, w.N, w.d, device=dev),
                torch.empty(w.B, w.H, w.N, w.dv, device=dev))
        ws = la.alloc_workspace(
            la.causal_backward_workspace_bytes(w.B, w.H, w.N, w.d, w.dv, w.dtype), dev)
        gam = head_decays(w.H).to(dev) if args.profile_case == "backward_decay" else None
        fn = lambda: la.backward_causal(q, k, v, dy, eps=w.eps, out=outs, workspace=ws, gamma=gam)
    else:
        q, k, v = make_qkv(w, device=dev, gen_device=dev)
        y = torch.empty(w.B, w.H, w.N, w.dv, device=dev)
        if w.mode == "noncausal":
            ws = la.alloc_workspace(la.noncausal_workspace_bytes(w.B, w.H, w.N, w.d, w.dv), dev)
            fn = lambda: la.forward_noncausal(q, k, v, eps=w.eps, out=y, workspace=ws)
        else:
            ws = la.alloc_workspace(la.causal_workspace_bytes(w.B, w.H, w.N, w.d, w.dv, w.dtype), dev)
            fn = lambda: la.forward_causal(q, k, v, eps=w.eps, out=y, workspace=ws)
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(3):
        fn()
    e1.record()
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": args.profile_case, "B": w.B, "H": w.H, "N": w.N,
                      "d": w.d, "dv": w.dv, "ms_per_call": e0.elapsed_time(e1) / 3}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-modes", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-case", choices=["causal", "long", "noncausal", "decode", "backward",
                                               "backward_decay",
                                               "causal_decay", "long_decay", "decode_decay",
                                               "gated"])
    ap.add_argument("--batch", type=int, default=0)
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.profile_case:
        profile_case(args)
        return
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        out = run_reference(args, world, rank)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    world, rank, local = dist_setup(args.gpus)
    out = run_ours(args, world, rank, local)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
