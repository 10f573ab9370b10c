#!/usr/bin/env python
"""Benchmark: SDPA forward and forward+backward TFLOP/s on one GB300.

Headline workload: bf16 GQA causal attention, B=2, Hq=32, Hkv=8, Lq=Lkv=4096, D=128,
scale=1/sqrt(128), logsumexp cached by the forward for the backward; inputs iid N(0,1)
from seed 3 (rank r adds 1000·r), rounded to bf16.  One step = sdpa_fwd + sdpa_bwd
(forward, δ pre-pass, dK/dV kernel, dQ kernel) through the C ABI, inputs resident in HBM.
FLOPs are algorithmic: 4·B·Hq·Lq·Lkv·D forward, 2.5× that backward, halved for causal.

Timing: W untimed warm-up steps, then exactly K steps, each bracketed by CUDA events on
the launching stream; L2 is flushed (a 256 MiB write) before every step, outside the
step's events.  Per-kernel durations come from the library's own event brackets
(sdpa_timing_*), recorded during a second pass of K steps (with the brackets on, the
backward runs its dK/dV and dQ kernels one after the other instead of concurrently).  SM
clocks and throttle reasons are sampled with nvidia-smi during both passes.  Also
measured in the same run: the same step end to end from pinned host buffers (copies
inside the timed region), the short-query (vector) path and the δ pre-pass against the
HBM roofline, attention masks, one line per (target workload, pass) with the oracle's
time and the GPU result's maximum errors against it, and the CPU oracle on a bounded
sample of the workload (the reported CPU baseline).

Multi-GPU (torchrun): every rank runs its own replica of the workload (the path needs no
exchange between GPUs); value = all ranks' FLOPs / the slowest rank's time; weak scaling.
`--impl reference` times the CPU oracle instead (rank 0 only), each step one query head
of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
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

WORKLOAD = dict(B=2, Hq=32, Hkv=8, Lq=4096, Lkv=4096, D=128)
CAUSAL = True
SEED = 3
METRIC = "SDPA fwd and fwd+bwd TFLOP/s on 1 GB300 & % of dense bf16 tensor peak"
WORKLOAD_NAME = "bf16 GQA causal SDPA fwd+bwd, B=2 Hq=32 Hkv=8 Lq=Lkv=4096 D=128"
SHORT_QUERY = dict(B=4, Hq=32, Hkv=8, Lq=8, Lkv=8192, D=128)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


def fwd_flops(B, Hq, Hkv, Lq, Lkv, D, causal):
    f = 4.0 * B * Hq * Lq * Lkv * D
    return f / 2 if causal else f


def slowest_rank(values, dist, device):
    """Element-wise maximum over the ranks of a list of times (ms): a job of replicas takes
    as long as its slowest replica.  Without a process group (dist None) the values come
    back as they are."""
    import torch
    t = torch.tensor(values, device=device, dtype=torch.float64)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def job_tflops(world, flops_per_step, steps, total_ms):
    """Whole-job throughput: the work of all `world` replicas over the slowest one's time."""
    return world * flops_per_step * steps / (total_ms / 1e3) / 1e12


def headline_config(world):
    """The `config` object of the headline line, shared by both arms (the GPU arm and the
    CPU oracle arm time the same workload)."""
    return {"workload": WORKLOAD_NAME, **WORKLOAD, "causal": CAUSAL,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": "flushed before every GPU step (256 MiB write, outside the step's events); "
                  "not applicable to the CPU oracle arm"}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_digest(name):
    p = os.path.join(ROOT, "scaled_dot_product_flash_gb300", "csrc", name)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def ncu_traffic(kernel):
    """DRAM bytes per launch from a committed ncu capture, or None if absent or stale."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f).get(kernel)
    if not d:
        return None
    if source_digest(d["source"]) != d["source_sha"]:
        return None
    return d["bytes_per_launch"]


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples, timestamped on the host."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(index), "-lms", "100"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.perf_counter(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        if not inside:  # region shorter than the sampling period: nearest sample after t0
            inside = [min(self.samples, key=lambda s: abs(s[0] - (t0 + t1) / 2))]
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for _, p in inside if num(p[1]) is not None]
        mx = [num(p[2]) for _, p in inside if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for _, p in inside for n, v in zip(names, p[5:9]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside),
                "power_w_max": max((num(p[3]) or 0.0) for _, p in inside)}


def cpu_baseline_sample(q, k, v, do, scale, heads):
    """Time the oracle (as it stands) on the first `heads` query heads of batch 0, one head
    at a time as the reference arm's steps do (the fp64 conversion of each head's inputs
    outside the timed part, like there), and return (TFLOP/s, seconds timed)."""
    import numpy as np  # noqa: F401
    import oracle
    from scaled_dot_product_flash_gb300.inputs import as_f64
    G = q.shape[1] // k.shape[1]
    dt = 0.0
    for h in range(heads):
        g = h // G
        qh, kg, vg, dh = (as_f64(t) for t in (q[0, h], k[0, g], v[0, g], do[0, h]))
        t0 = time.perf_counter()
        oracle.head_forward(qh, kg, vg, scale, CAUSAL, row_block=1024)
        oracle.head_backward(qh, kg, vg, dh, scale, CAUSAL, row_block=1024)
        dt += time.perf_counter() - t0
    W = WORKLOAD
    flops = 3.5 * fwd_flops(1, heads, 1, W["Lq"], W["Lkv"], W["D"], CAUSAL)
    return flops / dt / 1e12, dt


def run_reference(args):
    """CPU oracle arm: each step is one query head of the workload, fwd + bwd."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    import numpy as np
    import oracle
    from scaled_dot_product_flash_gb300.inputs import Shape, as_f64, draw
    W = WORKLOAD
    q, k, v, do = draw(Shape(**W), SEED, "bf16")
    scale = 1.0 / math.sqrt(W["D"])
    G = W["Hq"] // W["Hkv"]
    times = []
    for step in range(args.warmup + args.steps):
        h = step % W["Hq"]
        qh, kg, vg, dh = (as_f64(t) for t in (q[0, h], k[0, h // G], v[0, h // G], do[0, h]))
        t0 = time.perf_counter()
        oracle.head_forward(qh, kg, vg, scale, CAUSAL, row_block=1024)
        oracle.head_backward(qh, kg, vg, dh, scale, CAUSAL, row_block=1024)
        if step >= args.warmup:
            times.append(time.perf_counter() - t0)
    del np
    flops = 3.5 * fwd_flops(1, 1, 1, W["Lq"], W["Lkv"], W["D"], CAUSAL)
    ms = 1e3 * sum(times) / len(times)
    value = flops / (ms / 1e3) / 1e12
    cores = len(os.sched_getaffinity(0))
    sample = "one query head (Lq=Lkv=4096, D=128, causal) fwd+bwd per step, fp64 NumPy oracle"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": headline_config(args.gpus),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-(config, pass) lines")
    args = ap.parse_args()
    if args.impl == "reference":
        args.steps = args.steps or 20
        run_reference(args)
        return
    args.warmup = max(3, args.warmup)

    import torch
    import torch.distributed as dist
    from scaled_dot_product_flash_gb300 import _lib, api
    from scaled_dot_product_flash_gb300 import build as libbuild
    from scaled_dot_product_flash_gb300.inputs import Shape, draw

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0:
        libbuild.build()
    if world > 1:
        dist.barrier()
    _lib.load()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    W = WORKLOAD
    shape = Shape(**W)
    scale = 1.0 / math.sqrt(W["D"])
    q_h, k_h, v_h, do_h = draw(shape, SEED + 1000 * rank, "bf16")
    q, k, v, do = (t.to(dev) for t in (q_h, k_h, v_h, do_h))
    out = torch.empty_like(q)
    lse = torch.empty((W["B"], W["Hq"], W["Lq"]), device=dev, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(max(16, api.workspace_bytes(q, k)), device=dev, dtype=torch.uint8)
    flush = torch.empty(L2_FLUSH_BYTES, device=dev, dtype=torch.uint8)
    stream = torch.cuda.current_stream()

    def step():
        api.attention_forward(q, k, v, scale=scale, is_causal=CAUSAL, out=out, lse=lse)
        e_mid = torch.cuda.Event(enable_timing=True)
        e_mid.record(stream)
        api.attention_backward(q, k, v, out, do, lse, scale=scale, is_causal=CAUSAL,
                               workspace=ws, dq=dq, dk=dk, dv=dv)
        return e_mid

    for _ in range(args.warmup):
        flush.zero_()
        step()
    api.poll_status()
    # Default step count: about two seconds of timed work.
    if args.steps is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        torch.cuda.synchronize()
        args.steps = int(min(2000, max(10, 2000.0 / max(e0.elapsed_time(e1), 1e-3))))

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    mids = []
    barrier()
    launches0 = _lib.sdpa_launch_count()
    t0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        mids.append(step())
        ends[i].record(stream)
    barrier()
    t1 = time.perf_counter()
    launches = _lib.sdpa_launch_count() - launches0
    api.poll_status()
    clocks = sampler.summary(t0, t1) if sampler else None

    # Per-kernel durations: the same steps again with the library's per-kernel event
    # brackets on (the backward then runs dK/dV and dQ one after the other, so that each
    # bracket holds one kernel alone).
    _lib.sdpa_timing_reset()
    _lib.sdpa_timing_enable(True)
    tk0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        step()
    barrier()
    tk1 = time.perf_counter()
    _lib.sdpa_timing_enable(False)
    api.poll_status()
    kclocks = sampler.summary(tk0, tk1) if sampler else None

    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    fwd_ms = [s.elapsed_time(m) for s, m in zip(starts, mids)]
    total_ms, total_fwd_ms = slowest_rank([sum(step_ms), sum(fwd_ms)],
                                          dist if world > 1 else None, dev)
    ms_per_step = total_ms / args.steps
    F = fwd_flops(**W, causal=CAUSAL)
    step_flops = 3.5 * F
    value = job_tflops(world, step_flops, args.steps, total_ms)
    fwd_tflops = job_tflops(world, F, args.steps, total_fwd_ms)

    peaks, peak_src = load_peaks()
    bf16_peak = peaks["bf16_tflops"]
    bf16_sustained = peaks.get("bf16_tflops_sustained") or bf16_peak
    hbm_peak = peaks["hbm_gbs"]

    # Per-kernel achieved rates from the library's event brackets (same timed steps).
    kern = {}
    work = {"fwd": F, "dkdv": 2.0 * F, "dq": 0.5 * F}
    for name, kid in _lib.KERNELS.items():
        ms, n = _lib.sdpa_timing_read(kid)
        if n == 0:
            continue
        avg = ms / n
        entry = {"launches": n, "avg_ms": avg, "share": None}
        if name in work:
            entry["tflops"] = work[name] / (avg / 1e3) / 1e12
        if name == "delta":
            rows = W["B"] * W["Hq"] * W["Lq"]
            entry["gbs"] = (2 * rows * W["D"] * 2 + 4 * rows) / (avg / 1e3) / 1e9
        kern[name] = entry
    tot_k = sum(e["avg_ms"] * e["launches"] for e in kern.values())
    for e in kern.values():
        e["share"] = e["avg_ms"] * e["launches"] / tot_k if tot_k else None
    dom = max((n for n in kern if n in work), key=lambda n: kern[n]["avg_ms"] * kern[n]["launches"])
    path_is_tensor = _tensor_available()
    dom_src = {"fwd": "tc_fwd.cu", "dkdv": "tc_bwd.cu", "dq": "tc_bwd.cu"}[dom] \
        if path_is_tensor else "simt_kernels.cu"
    traffic = ncu_traffic(f"{dom}:{dom_src}")
    if path_is_tensor:
        # The dominant kernel's rate comes from the bracketed pass over the same seconds-long
        # run of back-to-back steps (the clock record shows the power cap engaged), so its
        # denominator is the sustained bf16 figure; the burst one is given beside it.
        roof = {"bound": "tensor", "achieved": kern[dom]["tflops"], "peak": bf16_sustained,
                "unit": "TFLOP/s", "frac": kern[dom]["tflops"] / bf16_sustained, "traffic": traffic,
                "kernel": dom,
                "peak_source": f"{peak_src} (sustained bf16: the kernel is timed inside a "
                               f"seconds-long run of steps)",
                "frac_of_burst_peak": kern[dom]["tflops"] / bf16_peak}
    else:
        alu_peak = alu_peak_tflops(clocks)
        roof = {"bound": "alu", "achieved": kern[dom]["tflops"], "peak": alu_peak,
                "unit": "TFLOP/s", "frac": kern[dom]["tflops"] / alu_peak, "traffic": traffic,
                "kernel": dom, "peak_source": "152 SMs x 128 fp32 FMA/clk x 2 x 2.07 GHz"}

    # End to end through the public API from pinned host buffers.
    e2e = run_e2e(torch, api, dev, stream, (q_h, k_h, v_h, do_h), scale, args.steps, step_flops,
                  world, barrier, dist if world > 1 else None)
    if sampler:
        sampler.stop()

    extras = {}
    configs = None
    if rank == 0:
        extras["short_query"] = run_short_query(torch, api, _lib, dev, stream, hbm_peak)
        extras["masked"] = run_masked(torch, api, dev, stream, bf16_peak)
        if not args.no_configs:
            configs = run_configs(torch, api, dev, stream, peaks, oracle_on=not args.no_cpu_baseline)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        heads = 16
        val, dt = cpu_baseline_sample(q_h, k_h, v_h, do_h, scale, heads)
        cpu = {"value": val, "unit": "TFLOP/s", "cores": len(os.sched_getaffinity(0)),
               "kind": "oracle",
               "sample": f"first {heads} query heads of batch 0, one head at a time (Lq=Lkv=4096, "
                         f"D=128, causal) fwd+bwd, fp64 NumPy oracle, {dt:.1f} s timed; the reference "
                         f"arm times the same per-head work, one head per step"}

    if world > 1:
        dist.barrier()
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": headline_config(world),
            "frac_of_bf16_peak": value / bf16_peak,
            # the headline steps run back to back for seconds under the power cap
            "frac_of_bf16_sustained_peak": value / bf16_sustained,
            "fwd": {"tflops": fwd_tflops, "ms": total_fwd_ms / args.steps,
                    "frac_of_bf16_peak": fwd_tflops / bf16_peak},
            "roofline": roof,
            "kernels": kern,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "clocks": clocks,
            "kernel_timing": {"how": "a second pass of the same steps with per-kernel event "
                                     "brackets on (dK/dV and dQ then serial)",
                              "clocks": kclocks},
            "configs": configs,
            "gpu_launches": launches,
            "peaks": {"source": peak_src, "bf16_tflops": bf16_peak,
                      "bf16_tflops_sustained": bf16_sustained, "hbm_gbs": hbm_peak},
            **extras,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def _tensor_available():
    """True when the tiled forward of the headline workload runs on the tensor-core path."""
    import torch
    from scaled_dot_product_flash_gb300 import _lib, api
    q = torch.zeros(1, 1, 128, 128, device="cuda", dtype=torch.bfloat16)
    try:
        with api.force_path(_lib.PATH_TENSOR):
            api.attention_forward(q, q, q, need_lse=False)
        return True
    except _lib.SdpaError:
        return False


def alu_peak_tflops(clocks):
    return 152 * 128 * 2 * 2.07e9 / 1e12


def run_e2e(torch, api, dev, stream, host_inputs, scale, steps, step_flops, world, barrier, dist):
    """Same step end to end from pinned host memory through the public API: every step
    copies q, k, v, dO host→device, runs forward + backward, and copies out, lse, dq, dk,
    dv device→host, all inside the timed region.  Steps are software-pipelined over three
    streams (copy in, compute, copy out) with two device buffer sets, so the copies of
    one step overlap the compute of its neighbours."""
    pin = [t.pin_memory() for t in host_inputs]
    W = WORKLOAD
    outs_h = [torch.empty_like(pin[0]).pin_memory(),
              torch.empty((W["B"], W["Hq"], W["Lq"]), dtype=torch.float32).pin_memory(),
              torch.empty_like(pin[0]).pin_memory(), torch.empty_like(pin[1]).pin_memory(),
              torch.empty_like(pin[2]).pin_memory()]
    sets = []
    for _ in range(2):
        ins = [torch.empty_like(t, device=dev) for t in pin]
        outs = [torch.empty_like(ins[0]), torch.empty((W["B"], W["Hq"], W["Lq"]), device=dev),
                torch.empty_like(ins[0]), torch.empty_like(ins[1]), torch.empty_like(ins[2])]
        ws = torch.empty(max(16, api.workspace_bytes(ins[0], ins[1])), device=dev, dtype=torch.uint8)
        sets.append((ins, outs, ws))
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    n = max(3, min(steps, 20))

    def run(count, start_ev=None, end_ev=None):
        comp_done, out_done = {}, {}
        if start_ev is not None:
            start_ev.record(s_in)
            s_cmp.wait_event(start_ev)
            s_out.wait_event(start_ev)
        for i in range(count):
            ins, outs, ws = sets[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(comp_done[i - 2])
                for d, h in zip(ins, pin):
                    d.copy_(h, non_blocking=True)
                in_done = torch.cuda.Event()
                in_done.record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(in_done)
                if i >= 2:
                    s_cmp.wait_event(out_done[i - 2])
                q, k, v, do = ins
                api.attention_forward(q, k, v, scale=scale, is_causal=CAUSAL, out=outs[0], lse=outs[1],
                                      stream=s_cmp)
                api.attention_backward(q, k, v, outs[0], do, outs[1], scale=scale, is_causal=CAUSAL,
                                       workspace=ws, dq=outs[2], dk=outs[3], dv=outs[4], stream=s_cmp)
                comp_done[i] = torch.cuda.Event()
                comp_done[i].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[i])
                for h, d in zip(outs_h, outs):
                    h.copy_(d, non_blocking=True)
                out_done[i] = torch.cuda.Event()
                out_done[i].record(s_out)
        if end_ev is not None:
            s_out.wait_event(comp_done[count - 1])
            s_out.wait_stream(s_in)
            end_ev.record(s_out)

    run(3)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    run(n, e0, e1)
    torch.cuda.synchronize()
    barrier()
    (ms,) = slowest_rank([e0.elapsed_time(e1)], dist, dev)
    h2d = sum(t.numel() * t.element_size() for t in pin)
    d2h = sum(t.numel() * t.element_size() for t in outs_h)
    return {"value": job_tflops(world, step_flops, n, ms), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms / n,
            "steps": n, "pipelined": "copy-in / compute / copy-out streams, 2 buffer sets"}


def run_short_query(torch, api, _lib, dev, stream, hbm_peak):
    """Short-query (vector) path, B=4 Hq=32 Hkv=8 Lkv=8192 D=128 bf16, Lq in {1, 4, 8}:
    HBM GB/s of forward and backward against the measured copy peak."""
    from scaled_dot_product_flash_gb300.inputs import Shape, draw
    res = {"workload": "bf16 short-query B=4 Hq=32 Hkv=8 Lkv=8192 D=128 non-causal, Lq in {1,4,8}",
           "timing": "median of 20 calls, L2 flushed before each"}
    flush = torch.empty(L2_FLUSH_BYTES, device=dev, dtype=torch.uint8)
    for lq in (1, 4, 8):
        S = dict(SHORT_QUERY, Lq=lq)
        q, k, v, do = (t.to(dev) for t in draw(Shape(**S), 4, "bf16"))
        scale = 1.0 / math.sqrt(S["D"])
        out, lse = api.attention_forward(q, k, v, scale=scale)
        dq, dk, dv = api.attention_backward(q, k, v, out, do, lse, scale=scale)
        fwd_t, bwd_t = [], []
        for i in range(23):
            flush.zero_()
            a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            a.record(stream)
            api.attention_forward(q, k, v, scale=scale, out=out, lse=lse)
            b.record(stream)
            flush.zero_()
            c0 = torch.cuda.Event(enable_timing=True)
            c0.record(stream)
            api.attention_backward(q, k, v, out, do, lse, scale=scale, dq=dq, dk=dk, dv=dv)
            c.record(stream)
            if i >= 3:
                fwd_t.append((a, b))
                bwd_t.append((c0, c))
        torch.cuda.synchronize()
        api.poll_status()
        fms = statistics.median(a.elapsed_time(b) for a, b in fwd_t)
        bms = statistics.median(a.elapsed_time(b) for a, b in bwd_t)
        kv = S["B"] * S["Hkv"] * S["Lkv"] * S["D"] * 2
        qb = S["B"] * S["Hq"] * S["Lq"] * S["D"] * 2
        rows = S["B"] * S["Hq"] * S["Lq"] * 4
        fwd_bytes = 2 * kv + 2 * qb + rows
        bwd_bytes = 4 * kv + 4 * qb + rows
        F = fwd_flops(**S, causal=False)
        res[f"Lq{lq}"] = {
            "fwd_ms": fms, "bwd_ms": bms,
            "fwd_gbs": fwd_bytes / (fms / 1e3) / 1e9, "bwd_gbs": bwd_bytes / (bms / 1e3) / 1e9,
            "fwd_frac_hbm": fwd_bytes / (fms / 1e3) / 1e9 / hbm_peak,
            "bwd_frac_hbm": bwd_bytes / (bms / 1e3) / 1e9 / hbm_peak,
            "fwd_tflops": F / (fms / 1e3) / 1e12, "bwd_tflops": 2.5 * F / (bms / 1e3) / 1e12,
            "algorithmic_bytes": {"fwd": fwd_bytes, "bwd": bwd_bytes}}
    return res


def run_masked(torch, api, dev, stream, bf16_peak):
    """Attention masks on the headline shape without the causal flag (every key tile is
    computed): forward + backward with no mask, a boolean key-padding mask [B, 1, 1, Lkv]
    (the last 10% of each batch's keys hidden) and an additive bf16 [Lq, Lkv] mask shared
    by every batch and head.  TFLOP/s count the work computed (non-causal FLOPs, backward
    2.5x the forward)."""
    from scaled_dot_product_flash_gb300.inputs import Shape, draw
    S = dict(WORKLOAD)
    res = {"workload": "bf16 B=2 Hq=32 Hkv=8 Lq=Lkv=4096 D=128, is_causal=False",
           "timing": "median of 10 forward+backward calls, L2 flushed before each"}
    q, k, v, do = (t.to(dev) for t in draw(Shape(**S), 5, "bf16"))
    scale = 1.0 / math.sqrt(S["D"])
    pad = torch.ones(S["B"], 1, 1, S["Lkv"], dtype=torch.bool, device=dev)
    pad[..., int(0.9 * S["Lkv"]):] = False
    gen = torch.Generator(device="cpu").manual_seed(6)
    add = torch.randn(S["Lq"], S["Lkv"], generator=gen).to(torch.bfloat16).to(dev)
    flush = torch.empty(L2_FLUSH_BYTES, device=dev, dtype=torch.uint8)
    F = fwd_flops(**S, causal=False)
    for name, mask in (("none", None), ("bool_key_padding", pad), ("additive_shared", add)):
        out, lse = api.attention_forward(q, k, v, scale=scale, attn_mask=mask)
        grads = api.attention_backward(q, k, v, out, do, lse, scale=scale, attn_mask=mask)
        times = []
        for i in range(13):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            api.attention_forward(q, k, v, scale=scale, attn_mask=mask, out=out, lse=lse)
            api.attention_backward(q, k, v, out, do, lse, scale=scale, attn_mask=mask,
                                   dq=grads[0], dk=grads[1], dv=grads[2])
            b.record(stream)
            if i >= 3:
                times.append((a, b))
        torch.cuda.synchronize()
        api.poll_status()
        ms = statistics.median(a.elapsed_time(b) for a, b in times)
        tf = 3.5 * F / (ms / 1e3) / 1e12
        res[name] = {"ms": ms, "tflops": tf, "frac_of_bf16_peak": tf / bf16_peak}
    return res


# Per-(config, pass) lines: the five target workloads (the short-query one at each Lq) and a
# head-dim-256 case.
# Seeds and the draw order follow the input recipe: one generator per workload; the
# short-query sub-runs draw one after another from default_rng(4).
CONFIGS = [
    ("C1 fp32 tiny", dict(B=1, Hq=2, Hkv=2, Lq=64, Lkv=64, D=32), "f32", False, 0),
    ("C2 fp32 B=8 H=8 L=128 D=64", dict(B=8, Hq=8, Hkv=8, Lq=128, Lkv=128, D=64), "f32", False, 1),
    ("C3 fp16 L=2048 D=64", dict(B=1, Hq=8, Hkv=8, Lq=2048, Lkv=2048, D=64), "f16", False, 2),
    ("C3 fp16 L=2048 D=64 causal", dict(B=1, Hq=8, Hkv=8, Lq=2048, Lkv=2048, D=64), "f16", True, 2),
    ("C4 bf16 GQA L=4096 D=128 causal", dict(WORKLOAD), "bf16", True, 3),
    ("C5a bf16 L=16384 D=128 causal", dict(B=1, Hq=16, Hkv=16, Lq=16384, Lkv=16384, D=128), "bf16",
     True, 4),
    # head dim 256 (the widest head the library serves; tensor-core forward and backward)
    ("D256 bf16 GQA L=4096 causal", dict(B=1, Hq=16, Hkv=4, Lq=4096, Lkv=4096, D=256), "bf16", True, 5),
]
# Oracle sample of the large workloads: whole (batch, KV head) groups.
ORACLE_GROUPS = {"C4 bf16 GQA L=4096 D=128 causal": [(1, 7)],
                 "C5a bf16 L=16384 D=128 causal": [(0, 11)],
                 "D256 bf16 GQA L=4096 causal": [(0, 3)]}


def _median_ms(torch, stream, fn, flush, n):
    times = []
    for i in range(n + 3):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        if i >= 3:
            times.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(x.elapsed_time(y) for x, y in times)


def _errors(dtype, got, ref):
    """Max errors of one comparison, in the units the tolerances use."""
    import numpy as np
    err = {"o_max_abs": float(np.max(np.abs(got["o"] - ref["o"]))),
           "lse_rel": float(np.max(np.abs(got["lse"] - ref["lse"]) /
                                   np.maximum(1.0, np.abs(ref["lse"]))))}
    for n in ("dq", "dk", "dv"):
        if dtype == "f32":
            err[n + "_max_abs"] = float(np.max(np.abs(got[n] - ref[n])))
        else:
            den = float(np.linalg.norm(ref[n])) or 1.0
            err[n + "_rel_frob"] = float(np.linalg.norm(got[n] - ref[n]) / den)
    return err


def _oracle_compare(name, S, dtype, causal, host, got, scale, groups):
    """Oracle on the whole workload (groups None) or on whole (batch, KV-head) groups;
    returns (seconds, sample description, max errors)."""
    import numpy as np
    import oracle
    from scaled_dot_product_flash_gb300.inputs import as_f64
    q, k, v, do = host
    G = S["Hq"] // S["Hkv"]
    if groups is None:
        t0 = time.perf_counter()
        qn, kn, vn, dn = (as_f64(t) for t in host)
        o, lse = oracle.sdpa_forward(qn, kn, vn, scale, causal)
        dq, dk, dv = oracle.sdpa_backward(qn, kn, vn, dn, scale, causal)
        dt = time.perf_counter() - t0
        ref = dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv)
        return dt, "whole workload", _errors(dtype, {n: as_f64(t) for n, t in got.items()}, ref)
    errs = {}
    dt = 0.0
    for b, g in groups:
        hs = slice(g * G, (g + 1) * G)
        t0 = time.perf_counter()
        kg, vg = as_f64(k[b, g]), as_f64(v[b, g])
        o = np.empty((G, S["Lq"], S["D"]))
        lse = np.empty((G, S["Lq"]))
        for t, h in enumerate(range(g * G, (g + 1) * G)):
            o[t], lse[t] = oracle.head_forward(as_f64(q[b, h]), kg, vg, scale, causal, row_block=1024)
        dq, dk, dv = oracle.group_backward(as_f64(q[b:b + 1]), as_f64(k[b:b + 1]), as_f64(v[b:b + 1]),
                                           as_f64(do[b:b + 1]), scale, causal, 0, g, row_block=1024)
        dt += time.perf_counter() - t0
        part = dict(o=as_f64(got["o"][b, hs]), lse=as_f64(got["lse"][b, hs]),
                    dq=as_f64(got["dq"][b, hs]), dk=as_f64(got["dk"][b, g]), dv=as_f64(got["dv"][b, g]))
        e = _errors(dtype, part, dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv))
        errs = {n: max(errs.get(n, 0.0), x) for n, x in e.items()}
    heads = G * len(groups)
    return dt, f"{len(groups)} whole (batch, KV head) group(s) = {heads} of {S['B'] * S['Hq']} query heads", errs


def run_configs(torch, api, dev, stream, peaks, oracle_on=True):
    """One entry per (config, pass): GPU time (median of CUDA-event brackets, L2 flushed
    before each call), TFLOP/s and the fraction of the bf16 peak (fp32 workloads also
    against the fp32 FMA peak of the CUDA cores), the oracle's time on this host's cores
    and the maximum errors of the GPU result against it."""
    import numpy as np
    from scaled_dot_product_flash_gb300.inputs import Shape, draw
    bf16_peak, hbm_peak = peaks["bf16_tflops"], peaks["hbm_gbs"]
    props = torch.cuda.get_device_properties(dev)
    sm_mhz = float(peaks.get("sm_max_mhz") or 2070.0)
    ffma_peak = props.multi_processor_count * 128 * 2 * sm_mhz * 1e6 / 1e12
    ffma_how = f"{props.multi_processor_count} SMs x 128 fp32 lanes x 2 FLOP (FMA) x {sm_mhz:.0f} MHz"
    cores = len(os.sched_getaffinity(0))
    flush = torch.empty(L2_FLUSH_BYTES, device=dev, dtype=torch.uint8)
    out = []
    jobs = []
    for name, S, dtype, causal, seed in CONFIGS:
        host = draw(Shape(**S), seed, dtype)
        jobs.append((name, S, dtype, causal, host))
    rng = np.random.default_rng(4)
    for lq in (1, 4, 8):
        S = dict(SHORT_QUERY, Lq=lq)
        jobs.append((f"C5b bf16 short query Lq={lq}", S, "bf16", False, draw(Shape(**S), 4, "bf16", rng=rng)))
    results = []
    for name, S, dtype, causal, host in jobs:
        q, k, v, do = (t.to(dev) for t in host)
        scale = 1.0 / math.sqrt(S["D"])
        o, lse = api.attention_forward(q, k, v, scale=scale, is_causal=causal)
        dq, dk, dv = api.attention_backward(q, k, v, o, do, lse, scale=scale, is_causal=causal)
        ws = torch.empty(max(16, api.workspace_bytes(q, k)), device=dev, dtype=torch.uint8)
        n = 20 if S["Lq"] * S["Lkv"] * S["Hq"] * S["B"] > (1 << 26) else 50

        def fwd():
            api.attention_forward(q, k, v, scale=scale, is_causal=causal, out=o, lse=lse)

        def both():
            fwd()
            api.attention_backward(q, k, v, o, do, lse, scale=scale, is_causal=causal, workspace=ws,
                                   dq=dq, dk=dk, dv=dv)
        fwd_ms = _median_ms(torch, stream, fwd, flush, n)
        both_ms = _median_ms(torch, stream, both, flush, n)
        api.poll_status()
        # results of one more clean call, copied to the host for the oracle comparison
        fwd()
        api.attention_backward(q, k, v, o, do, lse, scale=scale, is_causal=causal, dq=dq, dk=dk, dv=dv)
        api.poll_status()
        got = {n_: t.cpu() for n_, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
        results.append((name, S, dtype, causal, host, got, scale, fwd_ms, both_ms))
        del q, k, v, do, o, lse, dq, dk, dv, ws
    del flush
    torch.cuda.empty_cache()
    # The oracle runs after every GPU measurement, so it never competes with them.
    for name, S, dtype, causal, host, got, scale, fwd_ms, both_ms in results:
        F = fwd_flops(**S, causal=causal)
        orc = None
        if oracle_on:
            groups = ORACLE_GROUPS.get(name)
            dt, sample, errs = _oracle_compare(name, S, dtype, causal, host, got, scale, groups)
            full = dt if groups is None else dt * S["B"] * S["Hkv"] / len(groups)
            orc = {"seconds": dt, "sample": sample, "seconds_whole_workload": full,
                   "whole_workload_estimate": groups is not None, "cores": cores,
                   "max_errors": errs}
        short = name.startswith("C5b")
        for pas, ms, mult in (("fwd", fwd_ms, 1.0), ("fwd+bwd", both_ms, 3.5)):
            tf = mult * F / (ms / 1e3) / 1e12
            e = {"config": name, "shape": S, "dtype": dtype, "causal": bool(causal), "pass": pas,
                 "ms": ms, "tflops": tf, "frac_of_bf16_peak": tf / bf16_peak}
            if dtype == "f32":
                e["frac_of_fp32_ffma_peak"] = tf / ffma_peak
                e["fp32_ffma_peak_tflops"] = ffma_peak
                e["fp32_ffma_peak_how"] = ffma_how
            if short:
                kv = S["B"] * S["Hkv"] * S["Lkv"] * S["D"] * 2
                qb = S["B"] * S["Hq"] * S["Lq"] * S["D"] * 2
                rows = S["B"] * S["Hq"] * S["Lq"] * 4
                nbytes = (2 * kv + 2 * qb + rows) if pas == "fwd" else (2 * kv + 2 * qb + rows) + (4 * kv + 4 * qb + rows)
                e["gbs"] = nbytes / (ms / 1e3) / 1e9
                e["frac_of_hbm"] = e["gbs"] / hbm_peak
                e["algorithmic_bytes"] = nbytes
            if orc:
                e["oracle"] = orc
            out.append(e)
    return out


if __name__ == "__main__":
    main()
