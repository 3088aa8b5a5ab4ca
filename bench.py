"""Benchmark of the ring-attention hot path on GB300.

One step = one simulated rank of the large video context (432,000 tokens =
120 frames x 3,600 tokens, H = 4, d = 128, P = 8): the rank's 54,000 queries
against all 8 KV blocks in ring order, computed as one per-step fp32 partial
per ring step (one kernel launch over every (query tile pair, step) unit),
then the online-softmax merge of the 8 partials into bf16 O and fp32 LSE
(second launch).  Inputs are seeded synthetic bf16 N(0,1) tensors resident in
HBM; K and V (884 MB) exceed L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0).  --impl reference times the fp64 CPU oracle on
a bounded sample of the same workload instead.  With --gpus N > 1 (torchrun)
every rank runs an independent replica (the path has no data-parallel
collective on one node here); value = all ranks' work / max rank time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ring-attention fwd TFLOPS (bf16) & % dense BF16 peak; lse_merge HBM GB/s"
WORKLOAD = "c5"
WORKLOAD_DESC = ("one simulated rank of a 432,000-token video context (120 frames x 3,600 "
                 "tokens), H=4, d=128, P=8 contiguous, non-causal: 54,000 queries x 8 ring "
                 "blocks of 54,000 keys as per-step fp32 partials + lse_merge")


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target seconds of oracle work for the cpu_baseline sample")
    ap.add_argument("--kv-len", type=int, default=0,
                    help="smaller total sequence (same kernels and launch shape) for profiling")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--all-configs", action="store_true",
                    help="time the GPU path on every workload (c1..c5) and, in the same run, "
                         "the fp64 oracle on the host cores; one JSON line per workload")
    return ap.parse_args()


def _dist_init(n):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max_ms(ms, dist, device):
    """Max of a per-rank time over all ranks (the job is as slow as its slowest
    replica); identity without a process group."""
    if dist is None:
        return float(ms)
    import torch
    t = torch.tensor([float(ms)], device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            m = json.load(f)
        return {"hbm_gbs": m["hbm_gbs"], "bf16_tflops": m["bf16_tflops"],
                "bf16_tflops_sustained": m.get("bf16_tflops_sustained", m["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def _kernel_traffic(kernel_file, key):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    src = os.path.join(ROOT, "ring_attention_attn_gb300", "csrc", kernel_file)
    if not (os.path.exists(path) and os.path.exists(src)):
        return None
    with open(path) as f:
        t = json.load(f).get(key)
    if not t:
        return None
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return t["dram_bytes_per_launch"] if t.get("source_sha256_16") == digest else None


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"ra_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        loaded = [s for s in sm if smax and s > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def _workload(a):
    import dataclasses
    import synth
    w = synth.WORKLOADS[WORKLOAD]
    if a.kv_len:
        assert a.kv_len % (w.P * 2) == 0
        w = dataclasses.replace(w, S=a.kv_len)
    return w


def _cpu_baseline(seconds_target, quick_rows=4):
    """Time the fp64 oracle on sampled c5 query rows (host cores)."""
    import numpy as np
    import oracle
    import synth
    from ring_attention_attn_gb300 import accounting as acc

    w = synth.WORKLOADS[WORKLOAD]
    q, k, v = synth.make_qkv(w)
    per_row_flops = 4 * w.d * w.S
    # calibrate with a few rows, then size the sample to ~seconds_target
    rows = oracle.flat_rows(w.B, w.H, w.L, synth.sample_rows(w, quick_rows))
    t0 = time.perf_counter()
    oracle.attention(q, k, v, rows=rows)
    dt = time.perf_counter() - t0
    per_head = int(max(quick_rows, min(512, quick_rows * seconds_target / max(dt, 1e-3))))
    rows = oracle.flat_rows(w.B, w.H, w.L, synth.sample_rows(w, per_head))
    t0 = time.perf_counter()
    oracle.attention(q, k, v, rows=rows)
    dt = time.perf_counter() - t0
    flops = per_row_flops * len(rows)
    return {"value": flops / dt / 1e12, "unit": "TFLOPS", "cores": oracle.threads(),
            "kind": "oracle",
            "sample": f"{per_head} query rows per head x {w.B * w.H} heads of {WORKLOAD} "
                      f"(of {w.L}), all {w.S} keys, fp64; {dt:.2f} s",
            "seconds": dt, "full_workload_seconds_extrapolated":
                dt * (w.B * w.H * w.L) / len(rows)}


def run_reference(a, rank, world):
    if rank != 0:
        return
    import oracle
    import synth

    w = synth.WORKLOADS[WORKLOAD]
    q, k, v = synth.make_qkv(w)
    per_head = 24  # rows per head per step: ~27 GFLOP of fp64 per step
    all_rows = synth.sample_rows(w, per_head * (a.steps + a.warmup))
    flops_row = 4 * w.d * w.S
    times = []
    for i in range(a.warmup + a.steps):
        sel = all_rows[i * per_head:(i + 1) * per_head]
        rows = oracle.flat_rows(w.B, w.H, w.L, sel)
        t0 = time.perf_counter()
        oracle.attention(q, k, v, rows=rows)
        if i >= a.warmup:
            times.append(time.perf_counter() - t0)
    total = sum(times)
    flops = flops_row * per_head * w.B * w.H * a.steps
    value = flops / total / 1e12
    sample = (f"{per_head} query rows per head x {w.B * w.H} heads per step (of {w.L}), all "
              f"{w.S} keys, fp64 oracle on host cores")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
            "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
            "ms_per_step": 1e3 * total / a.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD_DESC, "B": w.B, "H": w.H, "S": w.S, "d": w.d,
                       "P": w.P, "rank": 0, "sample": sample},
            "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": oracle.threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(a, rank, world, local):
    import torch

    import synth
    import ring_attention_attn_gb300 as ra
    from ring_attention_attn_gb300 import accounting as acc

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    w = _workload(a)
    q, k, v = synth.make_qkv(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    n = w.P
    parts = torch.empty((n, w.B, w.H, w.L, w.d), dtype=torch.float32, device=dev)
    lparts = torch.empty((n, w.B, w.H, w.L), dtype=torch.float32, device=dev)
    out = torch.empty((w.B, w.H, w.L, w.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.H, w.L), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        ra.ring_attn_fwd_rank(qd, kd, vd, w.P, 0, out_fp32=True, out=parts, lse=lparts,
                              stream=stream)
        if ev is not None:
            ev[1].record(stream)
        ra.lse_merge(parts, lparts, out=out, lse_out=lse, stream=stream)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(a.warmup):
        step()
    torch.cuda.synchronize()
    if ra.ra_get_status() != 0:
        raise RuntimeError("device watchdog fired during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(a.steps)]
    clocks = ClockSampler(local)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(a.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    clock_info = clocks.stop()
    if dist is not None:
        dist.barrier()
    total_ms = t_start.elapsed_time(t_end)
    attn_ms = [e[0].elapsed_time(e[1]) for e in evs]
    merge_ms = [e[1].elapsed_time(e[2]) for e in evs]
    status = ra.ra_get_status()
    if status != 0:
        raise RuntimeError(f"device status {status}")
    total_ms = reduce_max_ms(total_ms, dist, dev)

    flops = acc.attention_flops(w.B * w.H, w.L, w.S, w.d)
    merge_bytes = acc.merge_bytes(n, w.B * w.H * w.L, w.d)
    value = world * flops * a.steps / (total_ms * 1e-3) / 1e12
    peaks = _peaks()
    attn_avg = statistics.mean(attn_ms)
    merge_avg = statistics.mean(merge_ms)
    attn_tflops = flops / (attn_avg * 1e-3) / 1e12
    merge_gbs = merge_bytes / (merge_avg * 1e-3) / 1e9
    # The attention kernel is timed in steps of tens of milliseconds, not in a
    # seconds-long loop: its denominator is the burst figure.  The ratio to
    # the sustained (power-capped, seconds-long) figure is reported beside it.
    peak_t = peaks["bf16_tflops"]

    # End to end through the public API with host buffers: every step copies
    # its inputs in from pinned host memory and its result out to pinned host
    # memory inside the timed region.  As a serving loop would, the copies run
    # on their own streams into double-buffered device tensors, so step i+1's
    # inputs arrive while step i computes and step i's result leaves while
    # step i+1 computes; the first step's copy-in and the last step's
    # copy-out are not hidden.
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    e2e_steps = max(1, a.steps)
    ins = [(qd, kd, vd), tuple(torch.empty_like(x) for x in (qd, kd, vd))]
    outs = [(out, lse), (torch.empty_like(out), torch.empty_like(lse))]
    hosts = [tuple(torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in o) for o in outs]
    copy_in = torch.cuda.Stream(dev)
    copy_out = torch.cuda.Stream(dev)

    def e2e_run(nsteps, t0=None, t1=None):
        ready = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        read = [torch.cuda.Event() for _ in range(2)]
        if t0 is not None:
            t0.record(copy_in)
        for i in range(nsteps):
            b = i % 2
            with torch.cuda.stream(copy_in):
                if i >= 2:
                    copy_in.wait_event(done[b])  # step i-2 has finished reading ins[b]
                for dst, src in zip(ins[b], (qh, kh, vh)):
                    dst.copy_(src, non_blocking=True)
                ready[b].record(copy_in)
            stream.wait_event(ready[b])
            if i >= 2:
                stream.wait_event(read[b])  # step i-2's result has left outs[b]
            ra.ring_attn_fwd_rank(*ins[b], w.P, 0, out_fp32=True, out=parts, lse=lparts,
                                  stream=stream)
            ra.lse_merge(parts, lparts, out=outs[b][0], lse_out=outs[b][1], stream=stream)
            done[b].record(stream)
            with torch.cuda.stream(copy_out):
                copy_out.wait_event(done[b])
                for dst, src in zip(hosts[b], outs[b]):
                    dst.copy_(src, non_blocking=True)
                read[b].record(copy_out)
        if t1 is not None:
            t1.record(copy_out)

    if a.no_e2e:
        e2e_steps = 0
    else:
        e2e_run(2)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e2e_clocks = ClockSampler(local)
    if e2e_steps:
        e2e_clocks.start()
        e2e_run(e2e_steps, e0, e1)
    torch.cuda.synchronize()
    e2e_clock_info = e2e_clocks.stop() if e2e_steps else None
    e2e_ms = e0.elapsed_time(e1) if e2e_steps else float("nan")
    if e2e_steps:
        e2e_ms = reduce_max_ms(e2e_ms, dist, dev)
        if ra.ra_get_status() != 0:
            raise RuntimeError("device watchdog fired during the end-to-end run")
    e2e_value = (world * flops * e2e_steps / (e2e_ms * 1e-3) / 1e12) if e2e_steps else None
    h2d = (q.numel() + k.numel() + v.numel()) * 2
    d2h = out.numel() * 2 + lse.numel() * 4

    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        cpu = _cpu_baseline(a.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": total_ms / a.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": WORKLOAD_DESC if not a.kv_len else
                       f"reduced profiling case of the same path: S={w.S}",
                       "B": w.B, "H": w.H, "S": w.S, "d": w.d,
                       "P": w.P, "rank": 0, "seq_len": w.S, "global_batch": w.B,
                       "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2 (K+V 884.7 MB per replica)"},
            "roofline": {"bound": "tensor", "achieved": attn_tflops, "peak": peak_t,
                         "unit": "TFLOP/s", "frac": attn_tflops / peak_t,
                         "traffic": _kernel_traffic("attn_fwd.cu", "ring_attn_kernel"),
                         "kernel": "ring_attn_kernel<128, fp32 partials>",
                         "peak_kind": f"bf16_tflops burst ({peaks['source']})",
                         "frac_of_sustained": attn_tflops / peaks["bf16_tflops_sustained"],
                         "sustained_peak": peaks["bf16_tflops_sustained"]},
            "merge": {"kernel": "lse_merge_kernel8<128, 1>", "bound": "hbm", "achieved": merge_gbs,
                      "peak": peaks["hbm_gbs"], "unit": "GB/s",
                      "frac": merge_gbs / peaks["hbm_gbs"], "bytes_per_launch": merge_bytes,
                      "ms": merge_avg,
                      "traffic": _kernel_traffic("merge.cu", "lse_merge_kernel")},
            "kernel_ms": {"ring_attn": attn_avg, "lse_merge": merge_avg},
            "clocks": clock_info,
            "e2e": {"value": e2e_value, "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "ms_per_step": (e2e_ms / e2e_steps) if e2e_steps else None,
                    "clocks": e2e_clock_info},
            "gpu_launches": 2 * a.steps,
        }
        if cpu is not None:
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def _gpu_ms(fn, reps, warmup=3):
    """Mean device time of fn() over `reps` back-to-back calls (CUDA events on
    the current stream, after `warmup` calls)."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def run_all_configs(a):
    """Every workload: the GPU path (inputs resident in HBM) and, in the same
    run, the fp64 oracle on the host cores (full for c1, c2, c4; stated row
    samples for c3 and c5), one JSON line each.  A baseline beside the GPU
    figure, not a target."""
    import numpy as np
    import torch

    import oracle
    import synth
    import ring_attention_attn_gb300 as ra
    from ring_attention_attn_gb300 import accounting as acc

    torch.cuda.set_device(0)
    peaks = _peaks()
    cores = oracle.threads()
    for name in ("c1", "c2", "c3", "c4", "c5"):
        w = synth.WORKLOADS[name]
        q, k, v = synth.make_qkv(w)
        BH = w.B * w.H
        if name == "c4":
            qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
            outs = (torch.empty_like(qd), torch.empty((w.B, w.H, w.S), device="cuda"),
                    torch.empty_like(qd), torch.empty((w.B, w.H, w.S), device="cuda"))
            ms = _gpu_ms(lambda: ra.factored_attn(qd, kd, vd, w.T, w.N, w.P, outs=outs), 20)
            sp, tp = acc.factored_flops(BH, w.T, w.N, w.d)
            flops = sp + tp
            t0 = time.perf_counter()
            oracle.factored(q, k, v, w.T, w.N, "spatial")
            oracle.factored(q, k, v, w.T, w.N, "temporal")
            cpu_s = time.perf_counter() - t0
            cpu_flops, sample = flops, "full (spatial + temporal)"
        elif name == "c5":
            qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
            parts = torch.empty((w.P, w.B, w.H, w.L, w.d), device="cuda")
            lp = torch.empty((w.P, w.B, w.H, w.L), device="cuda")
            out = torch.empty((w.B, w.H, w.L, w.d), dtype=torch.bfloat16, device="cuda")
            lse = torch.empty((w.B, w.H, w.L), device="cuda")

            def c5():
                ra.ring_attn_fwd_rank(qd, kd, vd, w.P, 0, out_fp32=True, out=parts, lse=lp)
                ra.lse_merge(parts, lp, out=out, lse_out=lse)
            ms = _gpu_ms(c5, 3)
            flops = acc.attention_flops(BH, w.L, w.S, w.d)
            per = synth.sample_rows(w, 128)
            rows = oracle.flat_rows(w.B, w.H, w.L, per)
            t0 = time.perf_counter()
            oracle.attention(q, k, v, rows=rows)
            cpu_s = time.perf_counter() - t0
            cpu_flops = 4 * w.d * w.S * len(rows)
            sample = f"128 query rows per head x {BH} heads (of {w.L}), all {w.S} keys"
        else:
            layout = 1 if w.causal else 0
            qd, kd, vd = (ra.ra_cp_shard(x.cuda(), w.P, layout) for x in (q, k, v))
            out = torch.empty_like(qd)
            lse = torch.empty((w.B, w.H, w.S), device="cuda")
            ms = _gpu_ms(lambda: ra.ring_attn_fwd(qd, kd, vd, w.P, causal=w.causal, out=out,
                                                  lse=lse), 20)
            flops = acc.attention_flops(BH, w.S, w.S, w.d, causal=w.causal)
            if name == "c3":
                per = synth.sample_rows(w, 512)
                rows = oracle.flat_rows(w.B, w.H, w.S, per)
                t0 = time.perf_counter()
                oracle.attention(q, k, v, rows=rows)
                cpu_s = time.perf_counter() - t0
                cpu_flops = 4 * w.d * w.S * len(rows)
                sample = f"512 query rows per head x {BH} heads (of {w.S}), all keys"
            else:
                t0 = time.perf_counter()
                oracle.attention(q, k, v, causal=w.causal)
                cpu_s = time.perf_counter() - t0
                cpu_flops, sample = flops, "full"
        if ra.ra_get_status() != 0:
            raise RuntimeError(f"device status after {name}")
        gpu_tflops = flops / (ms * 1e-3) / 1e12
        cpu_tflops = cpu_flops / cpu_s / 1e12
        line = {"workload": name, "config": dataclasses_dict(w), "gpu_ms": ms,
                "gpu_tflops": gpu_tflops, "gpu_frac_of_burst": gpu_tflops / peaks["bf16_tflops"],
                "algorithmic_gflop": flops / 1e9,
                "oracle": {"seconds": cpu_s, "tflops": cpu_tflops, "cores": cores,
                           "kind": "oracle", "sample": sample, "gflop": cpu_flops / 1e9,
                           "full_workload_seconds_extrapolated": cpu_s * flops / cpu_flops},
                "gpu_over_oracle": gpu_tflops / cpu_tflops, "peak_source": peaks["source"]}
        print(json.dumps(line), flush=True)


def dataclasses_dict(w):
    import dataclasses
    return {k: v for k, v in dataclasses.asdict(w).items() if k != "name"}


def main():
    a = _args()
    rank, world, local = _dist_init(a.gpus)
    if a.impl == "reference":
        run_reference(a, rank, world)
        return
    if a.all_configs:
        if rank == 0:
            run_all_configs(a)
        return
    run_ours(a, rank, world, local)


if __name__ == "__main__":
    main()
