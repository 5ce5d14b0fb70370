#!/usr/bin/env python
"""Benchmark of the attention forward hot path on GB300; prints one JSON line.

Default workload: causal attention forward, B=2, H=32, Nq=Nk=8192, d=128,
bf16 inputs drawn N(0,1) from fixed seeds, scale 1/sqrt(d).  The headline
`value` is its throughput in TFLOP/s, counting 4*B*H*Nq*Nk*d FLOPs halved for
causal, timed with CUDA events around every fa_fwd launch on the launching
stream, with the L2 cache flushed (a 256 MiB write) before each timed launch and
the device kept busy (a ~0.1 ms spin) while the host enqueues it.
The split-KV decode path (B=32, H=32, Nq=1, Nk=16384, d=128, bf16, 8 splits)
is timed the same way and reported under "decode" in GB/s, and its grouped-query
form (32 query heads over 8 K/V heads) under "decode_gqa".  A packed batch of 16
causal sequences of 256..8192 tokens goes under "varlen" (forward) and
"varlen_bwd" (its backward).  The backward of the default workload (fa_bwd, 2.5x
the forward's FLOPs) is reported under "bwd", and its FP8 (E4M3) forward from
pre-quantized inputs under "fp8" (with the quantization of Q, K, V timed beside
it).  "e2e" runs the default workload through fa_fwd_host: host buffers in and
out, the copies inside the timed region.  The fused forward at the benchmark's
other workloads is timed the same way and reported with its own roofline under
"cfg1" / "cfg1_causal" (B=1, H=1, N=128, d=64, fp16: one CTA, a latency case),
"cfg2" / "cfg2_causal" (B=4, H=16, N=1024, d=64, fp16), "cfg3_noncausal" (the
default shape without the mask) and "cfg4" (B=1, H=32, N=32768, d=128, bf16,
causal); the decode workload at 16 and 32 splits under "decode_s16" and
"decode_s32".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fa|reference]

--impl reference times the fp64 CPU oracle (the reference arm of this
benchmark) on a bounded sample of query rows of the same workload.
Under torchrun every rank runs an independent replica; rank 0 prints.
"""
from __future__ import annotations

import argparse
import hashlib
import itertools
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import attn_inputs  # noqa: E402

METRIC = "attention fwd TFLOP/s (fraction of GB300 dense BF16 peak); decode GB/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


# ----------------------------------------------------------------------------- helpers
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def dist_setup(n_gpus: int):
    """(rank, world, local_rank); initialises torch.distributed when launched by torchrun."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The largest value of x over all ranks (replica timings: the slowest rank decides)."""
    if world <= 1:
        return x
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


class ClockSampler:
    """Samples SM clock and throttle reasons with nvidia-smi while the timed region runs."""

    QUERY = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.rows = []
        self.proc = None
        self.thread = None
        self.active = False

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            if self.uuid and self.uuid not in parts[0] and parts[0] not in self.uuid:
                continue
            self.rows.append((time.time(), self.active, parts))

    def mark(self, active: bool):
        self.active = active

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self):
        rows = [r for r in self.rows if r[1]] or self.rows
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[2][1]) for r in rows if num(r[2][1]) is not None]
        smax = [num(r[2][2]) for r in rows if num(r[2][2]) is not None]
        power = [num(r[2][3]) for r in rows if num(r[2][3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[2][5:9]) if v.strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "reasons": reasons, "samples": len(rows)}


def device_uuid():
    try:
        u = torch.cuda.get_device_properties(torch.cuda.current_device()).uuid
        return "GPU-" + str(u)
    except Exception:  # noqa: BLE001
        return None


HOLD_CYCLES = 200_000  # ~0.1 ms of device time
# Idle time before each line after the headline.  A line that runs the GPU at its power
# cap for a while (the N = 32768 forward: 20 calls of 5 ms) leaves the clocks lowered
# for up to about a second; measured on GB300, the packed-batch forward took 1.30 ms
# per call right after it and 1.18 ms one second later.  Each line starts settled.
SETTLE_S = 1.0


def settle():
    torch.cuda.synchronize()
    time.sleep(SETTLE_S)


def time_calls(fn, steps: int, warmup: int, flush: torch.Tensor | None):
    """Per-call device milliseconds of fn() with CUDA events on the current stream.

    With `flush`, every timed call is preceded by an L2 flush (a 256 MiB write) and
    a short device-side spin (torch.cuda._sleep): the device is busy while the host
    enqueues the start event and the call, so the interval between the events holds
    the call's own kernels and no host-side launch gap.  Without `flush` (the
    end-to-end timing) the interval is whatever the call costs, host work included.
    """
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e0, e1 in evs:
        if flush is not None:
            flush.fill_(1)  # evicts the previous call's lines from L2
            torch.cuda._sleep(HOLD_CYCLES)
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    return [e0.elapsed_time(e1) for e0, e1 in evs]


# ----------------------------------------------------------------------------- CPU oracle timing
def oracle_rate(w: attn_inputs.Workload, wide, seconds: float, threads: int, seed: int = 0, max_rows: int = 1 << 16):
    """Time the fp64 oracle on sampled rows for about `seconds`; returns (TFLOP/s, rows, elapsed).

    `wide` is the workload widened to fp64 once (oracle.WidenedWorkload).  Each
    draw samples query rows (attn_inputs.sample_rows, linear in the count) and
    gathers them outside the timed region; the timed region is the oracle's
    arithmetic on those rows (every row over its full key range).  The draw
    grows (at most doubling) toward the size that fills the remaining time,
    capped at `max_rows` rows.
    """
    import oracle

    oracle.set_threads(threads)

    def flops_of(rows):
        vis = np.minimum(w.Nk, rows + (w.Nk - w.Nq) + 1) if w.causal else np.full(rows.shape, w.Nk)
        return float(4.0 * w.d * np.maximum(vis, 0).sum())

    BH = w.B * w.H
    n = max(threads, 8)
    t_total, f_total, rows_total = 0.0, 0.0, 0
    rnd = seed
    while True:
        pairs = attn_inputs.sample_rows(w.Nq, BH, n, seed=rnd)
        rnd += 1
        gathered = wide.gather(pairs)
        t0 = time.perf_counter()
        wide.rows(gathered, w.causal, w.scale)
        dt = time.perf_counter() - t0
        t_total += dt
        f_total += flops_of(gathered[1])
        rows_total += len(pairs)
        if t_total >= seconds:
            break
        n = int(min(2 * n, max(8.0, n * (seconds - t_total) / max(dt, 1e-3)), max_rows))
    return f_total / t_total / 1e12, rows_total, t_total


# ----------------------------------------------------------------------------- arms
def run_reference(args, rank, world):
    """The fp64 CPU oracle as the reference arm, on this arm's workload and metric."""
    if rank != 0:
        return
    w = attn_inputs.WORKLOADS[args.workload]
    threads = os.cpu_count() or 1
    q, k, v = attn_inputs.make_workload(w, "cpu")
    import oracle

    oracle.build()
    wide = oracle.WidenedWorkload(q, k, v)  # fp64 copies made once, before any timing
    del q, k, v
    budget = max(0.5, min(2.0, 150.0 / max(1, args.steps + args.warmup)))
    for i in range(args.warmup):
        oracle_rate(w, wide, budget * 0.25, threads, seed=10_000 + i)
    rates, times = [], []
    for i in range(args.steps):
        r, rows, dt = oracle_rate(w, wide, budget, threads, seed=20_000 + i)
        rates.append(r)
        times.append(dt)
    value = statistics.median(rates)
    sample = (f"each step: the fp64 oracle on about {budget:.1f} s of uniformly sampled query rows "
              f"(full key range per row) of {w.name}; inputs widened to fp64 once, before the timed steps")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * statistics.median(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w, flushed=False),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def workload_config(w: attn_inputs.Workload, flushed=True, parallelism="replicas"):
    return {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d, "dtype": w.dtype,
            "causal": w.causal, "scale": "1/sqrt(d)",
            "l2": "flushed before every timed launch (256 MiB write)" if flushed else "n/a",
            "parallelism": parallelism}


def run_fa(args, rank, world, local):
    import exact_attention_forward_03_gb300 as fa
    from exact_attention_forward_03_gb300 import build

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU; the CPU arm is --impl reference")
    build.build()
    fa.load_library()
    peaks, peak_src = load_peaks()
    dev = torch.device("cuda", torch.cuda.current_device())
    w = attn_inputs.WORKLOADS[args.workload]
    q, k, v = attn_inputs.make_workload(w, dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    sampler = ClockSampler(device_uuid())
    sampler.start()
    time.sleep(0.3)

    def call():
        fa.fwd(q, k, v, causal=w.causal, scale=w.scale, out=o, lse=lse)

    # The first launch of a kernel loads its module (lazy loading); keep that out of the
    # timed region's wall clock.
    call()
    torch.cuda.synchronize()

    # ---- timed region: fused forward
    barrier(world)
    torch.cuda.synchronize()
    sampler.mark(True)
    t_wall0 = time.perf_counter()
    ms = time_calls(call, args.steps, args.warmup, flush)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall0
    barrier(world)
    ms_mean = statistics.mean(ms)
    ms_max = max_over_ranks(ms_mean, world)
    status = fa.get_device_status()
    if status != fa.FA_OK:
        raise RuntimeError(f"device status {status} after the timed region")
    flops = w.flops()
    value = sum_over_ranks(flops, world) / (ms_max * 1e-3) / 1e12
    achieved = flops / (ms_mean * 1e-3) / 1e12
    launches = args.steps

    # ---- decode (split-KV + combine): multi-head, and grouped-query (several query heads per K/V head)
    def measure_decode(wd, fused=False, splits=None, inputs=None):
        splits = args.decode_splits if splits is None else splits
        dq, dk, dv = inputs if inputs is not None else attn_inputs.make_workload(wd, dev)
        do = torch.empty_like(dq)
        dl = torch.empty((wd.B, wd.H, wd.Nq), dtype=torch.float32, device=dev)
        ws = fa.splitkv_workspace(dq, dk, splits)

        def dcall():
            if fused:  # fa_fwd_gqa: a group's query heads as the rows of one tensor-core tile
                fa.fwd(dq, dk, dv, causal=False, scale=wd.scale, out=do, lse=dl)
            else:
                fa.fwd_splitkv(dq, dk, dv, causal=False, scale=wd.scale, num_splits=splits,
                               workspace=ws, out=do, lse=dl)

        settle()
        dms = time_calls(dcall, args.steps, args.warmup, flush)
        dmean = statistics.mean(dms)
        dbytes = wd.compulsory_bytes()
        gbs = dbytes / (dmean * 1e-3) / 1e9
        part_bytes = 2 * splits * wd.B * wd.H * wd.Nq * (wd.d + 1) * 4
        del dq, dk, dv, ws
        torch.cuda.empty_cache()
        return {"workload": wd.name, "entry_point": "fa_fwd_gqa" if fused else "fa_fwd_splitkv",
                "num_splits": None if fused else splits, "ms_per_call": dmean,
                "value": sum_over_ranks(dbytes, world) / (max_over_ranks(dmean, world) * 1e-3) / 1e9,
                "unit": "GB/s",
                "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": gbs / peaks["hbm_gbs"], "traffic": None,
                             "note": f"compulsory bytes (Q, K, V read, O, LSE written) per call; peak {peak_src}"
                                     + ("" if fused else "; split-partial traffic (written and re-read by the "
                                        f"combine) excluded: {part_bytes} bytes per call")}}

    # ---- the fused forward at every other workload of the benchmark (one fa_fwd launch per call)
    def measure_fwd(wname):
        wf = attn_inputs.WORKLOADS[wname]
        fq, fk, fv = attn_inputs.make_workload(wf, dev)
        fo = torch.empty_like(fq)
        fl = torch.empty((wf.B, wf.H, wf.Nq), dtype=torch.float32, device=dev)

        def fcall():
            fa.fwd(fq, fk, fv, causal=wf.causal, scale=wf.scale, out=fo, lse=fl)

        settle()
        fms = time_calls(fcall, args.steps, args.warmup, flush)
        fmean = statistics.mean(fms)
        if fa.get_device_status() != fa.FA_OK:
            raise RuntimeError(f"device status not ok after {wname}")
        fflops = wf.flops()
        ach = fflops / (fmean * 1e-3) / 1e12
        kern = f"fa_fwd_kernel<{wf.d},{wf.dtype}>"
        del fq, fk, fv, fo, fl
        torch.cuda.empty_cache()
        return {"workload": wf.name, "entry_point": "fa_fwd", "ms_per_call": fmean, "us_per_call": 1e3 * fmean,
                "ms_min": min(fms), "value": sum_over_ranks(fflops, world) / (max_over_ranks(fmean, world) * 1e-3) / 1e12,
                "unit": "TFLOP/s", "flops_per_call": fflops, "grid_ctas": wf.B * wf.H * ((wf.Nq + 127) // 128),
                "roofline": {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                             "frac": ach / peaks["bf16_tflops"],
                             "frac_of_sustained": ach / peaks["bf16_tflops_sustained"],
                             "traffic": captured_traffic(kern, wf.name), "kernel": kern,
                             "note": "fp16 and bf16 share the dense 16-bit tensor rate; peak "
                                     f"{peak_src} bf16 burst"}}

    workload_lines = {}
    if not args.no_configs:
        for key, wname in (("cfg1", "tiny_d64_f16"), ("cfg1_causal", "tiny_d64_f16_causal"),
                           ("cfg2", "b4h16_n1024_d64_f16"), ("cfg2_causal", "b4h16_n1024_d64_f16_causal"),
                           ("cfg3_noncausal", "b2h32_n8192_d128_bf16"),
                           ("cfg4", "b1h32_n32768_d128_bf16_causal")):
            if wname != w.name:
                workload_lines[key] = measure_fwd(wname)
                launches += args.steps

    # ---- packed variable-length batch (fa_fwd_varlen)
    varlen = varlen_bwd = None
    if not args.no_varlen:
        vw = attn_inputs.VARLEN_WORKLOAD
        lens = attn_inputs.varlen_lengths(vw["num_seqs"], vw["lo"], vw["hi"], vw["seed"])
        total = sum(lens)
        # packed [total, H, d] tensors: the [B, H, N, d] recipe with B = 1, H = total, N = H
        vq = attn_inputs.make_qkv(1, total, vw["H"], 1, vw["d"], vw["dtype"], vw["seed"], dev)[0][0]
        _, vk, vv = attn_inputs.make_qkv(1, total, 1, vw["H"], vw["d"], vw["dtype"], vw["seed"] + 5, dev)
        vk, vv = vk[0], vv[0]
        cu = torch.tensor([0] + list(itertools.accumulate(lens)), dtype=torch.int32, device=dev)
        vo = torch.empty_like(vq)
        vl = torch.empty((vw["H"], total), dtype=torch.float32, device=dev)
        vws = torch.empty(fa.fwd_varlen_workspace_bytes(len(lens), total), dtype=torch.uint8, device=dev)

        def vcall():
            # fa_fwd_varlen_ws: the work-list launch, then the forward over row blocks that hold rows
            fa.fwd_varlen(vq, vk, vv, cu, cu, causal=vw["causal"], out=vo, lse=vl, workspace=vws)

        settle()
        vms = time_calls(vcall, args.steps, args.warmup, flush)
        launches += 2 * args.steps
        vmean = statistics.mean(vms)
        vflops = sum(4.0 * vw["H"] * n * n * vw["d"] / (2.0 if vw["causal"] else 1.0) for n in lens)
        varlen = {"workload": vw["name"], "entry_point": "fa_fwd_varlen_ws", "launches_per_call": 2,
                  "lengths": lens, "total_tokens": total, "ms_per_call": vmean,
                  "value": sum_over_ranks(vflops, world) / (max_over_ranks(vmean, world) * 1e-3) / 1e12,
                  "unit": "TFLOP/s", "flops_per_call": vflops,
                  "roofline": {"bound": "tensor", "achieved": vflops / (vmean * 1e-3) / 1e12,
                               "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                               "frac": vflops / (vmean * 1e-3) / 1e12 / peaks["bf16_tflops"], "traffic": None}}
        if not args.no_bwd:
            # the backward of the same packed batch (fa_bwd_varlen: plan, preprocess, main kernel, dQ conversion)
            vg = attn_inputs.make_dout(1, total, vw["H"], vw["d"], vw["dtype"], vw["seed"], dev)[0]
            vdq, vdk, vdv = torch.empty_like(vq), torch.empty_like(vk), torch.empty_like(vv)
            vws = torch.empty(fa.bwd_varlen_workspace_bytes(len(lens), total, total, vw["H"], vw["d"]), dtype=torch.uint8,
                              device=dev)
            vcall()

            def vbcall():
                fa.bwd_varlen(vq, vk, vv, vo, vg, vl, cu, cu, max(lens), causal=vw["causal"], dq=vdq, dk=vdk, dv=vdv,
                              workspace=vws)

            settle()
            vbms = time_calls(vbcall, args.steps, args.warmup, flush)
            launches += 5 * args.steps
            vbmean = statistics.mean(vbms)
            vbflops = 2.5 * vflops
            varlen_bwd = {"workload": vw["name"], "entry_point": "fa_bwd_varlen", "launches_per_call": 5,
                          "ms_per_call": vbmean,
                          "value": sum_over_ranks(vbflops, world) / (max_over_ranks(vbmean, world) * 1e-3) / 1e12,
                          "unit": "TFLOP/s", "flops_per_call": vbflops,
                          "roofline": {"bound": "tensor", "achieved": vbflops / (vbmean * 1e-3) / 1e12,
                                       "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                                       "frac": vbflops / (vbmean * 1e-3) / 1e12 / peaks["bf16_tflops"],
                                       "traffic": None,
                                       "note": "whole call (five launches) timed; FLOPs 2.5x the forward's"}}
            if fa.get_device_status() != fa.FA_OK:
                raise RuntimeError("device status not ok after the variable-length backward")
            del vg, vdq, vdk, vdv, vws
        del vq, vk, vv, vo, vl
        torch.cuda.empty_cache()

    # ---- backward (fa_bwd: preprocess, main K/V-block kernel, dQ conversion) on the same workload
    bwd = None
    if not args.no_bwd:
        gout = attn_inputs.make_dout(w.B, w.H, w.Nq, w.d, w.dtype, w.seed, dev)
        fa.fwd(q, k, v, causal=w.causal, scale=w.scale, out=o, lse=lse)
        gq, gk, gv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        gws = torch.empty(fa.bwd_workspace_bytes(w.B, w.H, w.Nq, w.d), dtype=torch.uint8, device=dev)

        def bcall():
            fa.bwd(q, k, v, o, gout, lse, causal=w.causal, scale=w.scale, dq=gq, dk=gk, dv=gv, workspace=gws)

        settle()
        bms = time_calls(bcall, args.steps, args.warmup, flush)
        launches += 3 * args.steps
        bmean = statistics.mean(bms)
        bflops = 2.5 * flops  # five products of the forward's size against the forward's two
        bwd = {"workload": w.name, "entry_point": "fa_bwd", "launches_per_call": 3, "ms_per_call": bmean,
               "ms_min": min(bms), "value": sum_over_ranks(bflops, world) / (max_over_ranks(bmean, world) * 1e-3) / 1e12,
               "unit": "TFLOP/s", "flops_per_call": bflops,
               "roofline": {"bound": "tensor", "achieved": bflops / (bmean * 1e-3) / 1e12, "peak": peaks["bf16_tflops"],
                            "unit": "TFLOP/s", "frac": bflops / (bmean * 1e-3) / 1e12 / peaks["bf16_tflops"],
                            "traffic": captured_traffic("fa_bwd_call<128,bf16>", w.name),
                            "note": "whole call (three launches) timed; FLOPs 2.5x the forward's; traffic = DRAM bytes "
                                    "of the three launches of one call"}}
        status = fa.get_device_status()
        if status != fa.FA_OK:
            raise RuntimeError(f"device status {status} after the backward")
        del gout, gq, gk, gv, gws
        torch.cuda.empty_cache()

    # ---- FP8 (E4M3) forward of the same workload from pre-quantized inputs
    fp8 = None
    if not args.no_fp8 and w.d == 128:
        q8, qs = fa.fp8_quantize(q)
        k8, ks = fa.fp8_quantize(k)
        v8t, vs = fa.fp8_quantize(v, transpose=True)
        o8 = torch.empty_like(o)

        def qcall():
            fa.fp8_quantize(q, out=q8, scales=qs)
            fa.fp8_quantize(k, out=k8, scales=ks)
            fa.fp8_quantize(v, transpose=True, out=v8t, scales=vs)

        def fcall():
            fa.fwd_fp8(q8, qs, k8, ks, v8t, vs, causal=w.causal, scale=w.scale, out_dtype=q.dtype, out=o8, lse=lse)

        settle()
        fms = time_calls(fcall, args.steps, args.warmup, flush)
        qms = time_calls(qcall, max(3, min(args.steps, 20)), args.warmup, flush)
        launches += args.steps + 3 * max(3, min(args.steps, 20))
        fmean = statistics.mean(fms)
        qbytes = 3.0 * q.numel() * (q.element_size() + 1) + 3.0 * w.B * w.H * ((w.Nq + 127) // 128) * 4
        fpeak = 2.0 * peaks["bf16_tflops"]  # E4M3 dense rate = 2x bf16 (nominal 4.5 vs 2.25 PFLOP/s)
        fach = flops / (fmean * 1e-3) / 1e12
        fp8 = {"workload": w.name, "entry_point": "fa_fwd_fp8", "ms_per_call": fmean, "ms_min": min(fms),
               "value": sum_over_ranks(flops, world) / (max_over_ranks(fmean, world) * 1e-3) / 1e12, "unit": "TFLOP/s",
               "quantize_ms_per_call": statistics.mean(qms),
               "quantize_roofline": {"bound": "hbm", "unit": "GB/s", "peak": peaks["hbm_gbs"],
                                     "achieved": qbytes / (statistics.mean(qms) * 1e-3) / 1e9,
                                     "frac": qbytes / (statistics.mean(qms) * 1e-3) / 1e9 / peaks["hbm_gbs"],
                                     "note": "fa_fp8_quantize of Q, K, V: 16-bit inputs read, E4M3 codes and "
                                             "per-block scales written (compulsory bytes)"},
               "roofline": {"bound": "tensor", "achieved": fach, "peak": fpeak, "unit": "TFLOP/s", "frac": fach / fpeak,
                            "traffic": captured_traffic("fa_fwd_fp8_kernel<bf16>", w.name),
                            "note": "inputs quantized beforehand (fa_fp8_quantize of Q, K, V timed separately as "
                                    "quantize_ms_per_call); peak = 2 x measured bf16 (the E4M3/bf16 nominal ratio)"}}
        del q8, k8, v8t, o8
        torch.cuda.empty_cache()

    decode = decode_gqa = None
    if not args.no_decode:
        del q, k, v
        torch.cuda.empty_cache()
        wdec = attn_inputs.WORKLOADS[args.decode_workload]
        dec_in = attn_inputs.make_workload(wdec, dev)
        decode = measure_decode(wdec, inputs=dec_in)
        launches += 2 * args.steps
        for sp in (8, 16, 32):  # the split count against the HBM roofline (`decode` is --decode-splits)
            if sp != args.decode_splits:
                workload_lines[f"decode_s{sp}"] = measure_decode(wdec, splits=sp, inputs=dec_in)
                launches += 2 * args.steps
        del dec_in
        torch.cuda.empty_cache()
        if args.decode_gqa_workload:
            decode_gqa = measure_decode(attn_inputs.WORKLOADS[args.decode_gqa_workload], fused=True)
            launches += args.steps
        q, k, v = attn_inputs.make_workload(w, dev)
    sampler.mark(False)
    sampler.stop()
    clocks = sampler.summary()

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        qh, kh, vh = (t.to("cpu").pin_memory() for t in (q, k, v))
        oh = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        lh = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
        ews = torch.empty(fa.fwd_host_workspace_bytes(w.B, w.H, w.kv_heads, w.Nq, w.Nk, w.d), dtype=torch.uint8,
                          device=dev)
        nchunks = 8

        def ecall():
            # one fa_fwd_host call: pinned host inputs in, pinned host outputs back, the
            # copies of one chunk of heads overlapped with the compute of the previous one
            fa.fwd_host(qh, kh, vh, causal=w.causal, scale=w.scale, out=oh, lse=lh, num_chunks=nchunks,
                        workspace=ews, synchronize=False)

        esteps = max(3, min(args.steps, 20))
        ems = time_calls(ecall, esteps, max(1, min(args.warmup, 3)), None)
        launches += esteps * min(nchunks, w.B * w.kv_heads)
        emean = max_over_ranks(statistics.mean(ems), world)
        h2d = qh.numel() * qh.element_size() + 2 * kh.numel() * kh.element_size()
        d2h = oh.numel() * oh.element_size() + lh.numel() * 4
        # The host link's bound for one step: the same byte counts copied host->device and
        # device->host at once on two streams, with no compute.
        lin, lout = torch.empty(h2d, dtype=torch.uint8, device=dev), torch.empty(d2h, dtype=torch.uint8, device=dev)
        hin = torch.empty(h2d, dtype=torch.uint8, pin_memory=True)
        hout = torch.empty(d2h, dtype=torch.uint8, pin_memory=True)
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

        def link_step():
            s_in.wait_stream(torch.cuda.current_stream())
            s_out.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s_in):
                lin.copy_(hin, non_blocking=True)
            with torch.cuda.stream(s_out):
                hout.copy_(lout, non_blocking=True)
            torch.cuda.current_stream().wait_stream(s_in)
            torch.cuda.current_stream().wait_stream(s_out)

        lms = statistics.median(time_calls(link_step, 5, 1, None))
        e2e = {"value": sum_over_ranks(flops, world) / (emean * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": emean, "steps": esteps, "entry_point": "fa_fwd_host",
               "link_bound_ms": lms, "frac_of_link_bound": lms / emean,
               "note": f"host (page-locked) buffers in and out; {nchunks} chunks of heads, copies overlapped with "
                       "the kernels of the previous chunk; link_bound_ms = the step's host->device and "
                       "device->host bytes copied at once with no compute"}
        del ews, lin, lout, hin, hout

    # ---- the oracle on this machine's host cores (rank 0, N=1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle

        threads = os.cpu_count() or 1
        wide = oracle.WidenedWorkload(q, k, v)  # fp64 host copies, made before the timing
        rate, rows, secs = oracle_rate(w, wide, args.cpu_seconds, threads)
        rate1, rows1, secs1 = oracle_rate(w, wide, max(1.0, args.cpu_seconds / 4), 1, seed=30_000)
        oracle.set_threads(threads)
        del wide
        cpu = {"value": rate, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"{rows} uniformly sampled query rows of {w.name} (full key range each), {secs:.1f} s "
                         "of oracle arithmetic (inputs widened to fp64 once, outside the timing)",
               "extrapolated_full_oracle_s": w.flops() / (rate * 1e12),
               "single_core": {"value": rate1, "unit": "TFLOP/s", "cores": 1, "rows": rows1, "seconds": secs1,
                               "extrapolated_full_oracle_s": w.flops() / (rate1 * 1e12)}}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f16", "data": "synthetic",
        "config": workload_config(w),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / peaks["bf16_tflops"],
                     "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                     "traffic": args.traffic if args.traffic is not None else captured_traffic("fa_fwd_kernel<128,bf16>", w.name),
                     "peak_source": peak_src,
                     "kernel": "fa_fwd_kernel<128,bf16>", "flops_per_launch": flops},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clocks, "decode": decode,
        "decode_gqa": decode_gqa, "varlen": varlen, "varlen_bwd": varlen_bwd, "bwd": bwd, "fp8": fp8,
        **workload_lines,
        "wall_s_fwd_timed": wall, "ms_fwd_min": min(ms), "ms_fwd_median": statistics.median(ms),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def captured_traffic(kernel, workload):
    """DRAM bytes (read + write) per launch of `kernel` on `workload` from the ncu
    capture summarised under profiles/, or None when there is none or when the
    kernel's sources changed since the counters were taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            entry = json.load(f).get(kernel)
        if entry is None or entry.get("workload") != workload:
            return None
        h = hashlib.sha256()
        for rel in entry["source_files"]:
            with open(os.path.join(ROOT, rel), "rb") as f:
                h.update(f.read())
        if h.hexdigest() != entry["source_sha256"]:
            return None
        return float(entry["dram_bytes_read"] + entry["dram_bytes_write"])
    except (OSError, ValueError, KeyError):
        return None


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["fa", "reference"], default="fa")
    ap.add_argument("--workload", default="b2h32_n8192_d128_bf16_causal", choices=sorted(attn_inputs.WORKLOADS))
    ap.add_argument("--decode-workload", default="decode_b32h32_nk16384_d128_bf16")
    ap.add_argument("--decode-splits", type=int, default=8)
    ap.add_argument("--decode-gqa-workload", default="decode_b32h32kv8_nk16384_d128_bf16",
                    help="grouped-query decode workload reported under decode_gqa ('' to skip)")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the forward at the other workloads (cfg1, cfg1_causal, cfg2, cfg2_causal, "
                         "cfg3_noncausal, cfg4)")
    ap.add_argument("--no-varlen", action="store_true")
    ap.add_argument("--no-bwd", action="store_true")
    ap.add_argument("--no-fp8", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the fused kernel from an ncu capture (reported as roofline.traffic)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up calls, whatever was asked
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_fa(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
