"""Per-entry-point throughput on the workloads of the ring-attention path.

Times every public entry point with CUDA events on the current stream (inputs
resident in HBM, 3 warm-up calls, then `reps` calls back to back between two
events: the mean, launch gaps hidden as in a real pipeline) and prints one
JSON line per path with its algorithmic throughput and roofline fraction
against MEASURED_PEAKS.json (bf16 dense burst peak for contractions, HBM copy
bandwidth for permutations and merges).  With --graph each line also
carries the per-call time of the same calls captured in one CUDA graph and
replayed (`graph_ms`: no host submission between calls, so for the short
workloads it is the device time that back-to-back calls hide behind the
host's per-call cost).  Usage:

    python -m ring_attention_attn_gb300.measure [--path NAME ...] [--reps N] [--graph]

Paths: shard, transpose, merge, ring_c1, ring_c2, ring_c3, rank_c5, factored_c4,
factored_c4_unfolded, overlap_c3, overlap_c3_stream, ulysses_c3, allgather_c3,
reducescatter_c3, bwd_c3.
"""
from __future__ import annotations

import argparse
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            m = json.load(f)
        return {"hbm_gbs": m["hbm_gbs"], "bf16_tflops": m["bf16_tflops"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


_GRAPH = {"on": False, "ms": None}


def _time(fn, reps):
    import torch
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    _GRAPH["ms"] = _time_graph(fn, reps) if _GRAPH["on"] else None
    return e0.elapsed_time(e1) / reps


def _time_graph(fn, reps):
    """Mean per-call time of `reps` calls captured in one CUDA graph and
    replayed three times; None when the calls cannot be captured."""
    import torch
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(2):
                fn()
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(reps):
                fn()
        g.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(3):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / (3 * reps)
    except RuntimeError:
        torch.cuda.synchronize()
        return None


def _rand(shape, gen):
    import torch
    return torch.randn(shape, device="cuda", generator=gen).bfloat16()


def run(paths, reps, graph=False):
    import torch
    _GRAPH["on"] = graph

    sys.path.insert(0, ROOT)
    import ring_attention_attn_gb300 as ra
    from ring_attention_attn_gb300 import accounting as acc

    pk = _peaks()
    gen = torch.Generator(device="cuda").manual_seed(0)
    out = []

    def emit(path, ms, work, unit, bound, **extra):
        if unit == "TFLOP/s":
            val, peak = work / ms / 1e9, pk["bf16_tflops"]
        else:
            val, peak = work / ms / 1e6, pk["hbm_gbs"]
        line = {"path": path, "ms": ms, "achieved": val, "unit": unit, "bound": bound,
                "peak": peak, "frac": val / peak, "peak_source": pk["source"], **extra}
        if _GRAPH["on"]:
            gms = _GRAPH["ms"]
            line["graph_ms"] = gms
            line["graph_achieved"] = (val * ms / gms) if gms else None
        print(json.dumps(line), flush=True)
        out.append(line)

    def qkv(B, H, S, d):
        return (_rand((B, H, S, d), gen) for _ in range(3))

    for path in paths:
        if path == "shard":
            x = _rand((1, 4, 4096 * 64, 128), gen)
            y = torch.empty_like(x)
            ms = _time(lambda: ra.ra_cp_shard(x, 8, 1, out=y), reps)
            emit(path, ms, acc.shard_bytes(4, 4096 * 64, 128), "GB/s", "hbm", layout="zigzag P=8")
        elif path == "transpose":
            x = _rand((1, 24, 43200, 128), gen)
            y = torch.empty_like(x)
            ms = _time(lambda: ra.ra_frame_transpose(x, 48, 900, out=y), reps)
            emit(path, ms, acc.shard_bytes(24, 43200, 128), "GB/s", "hbm", shape="T=48 N=900")
        elif path == "merge":
            o = torch.randn((8, 216000, 128), device="cuda", generator=gen) * 0.25
            l = torch.randn((8, 216000), device="cuda", generator=gen)
            mo = torch.empty((216000, 128), dtype=torch.bfloat16, device="cuda")
            ml = torch.empty(216000, device="cuda")
            ms = _time(lambda: ra.lse_merge(o, l, out=mo, lse_out=ml), reps)
            emit(path, ms, acc.merge_bytes(8, 216000, 128), "GB/s", "hbm", n=8)
        elif path.startswith("ring_c"):
            B, H, S, d, P, causal = {"ring_c1": (1, 2, 1024, 64, 4, False),
                                     "ring_c2": (1, 4, 4096, 64, 2, True),
                                     "ring_c3": (1, 24, 14400, 128, 4, False)}[path]
            q, k, v = qkv(B, H, S, d)
            o = torch.empty_like(q)
            lse = torch.empty((B, H, S), device="cuda")
            ms = _time(lambda: ra.ring_attn_fwd(q, k, v, P, causal=causal, out=o, lse=lse), reps)
            emit(path, ms, acc.attention_flops(B * H, S, S, d, causal=causal), "TFLOP/s",
                 "tensor")
        elif path == "rank_c5":
            H, S, d, P = 4, 432000, 128, 8
            L = S // P
            q = _rand((1, H, L, d), gen)
            k, v = _rand((1, H, S, d), gen), _rand((1, H, S, d), gen)
            parts = torch.empty((P, 1, H, L, d), device="cuda")
            lp = torch.empty((P, 1, H, L), device="cuda")
            ms = _time(lambda: ra.ring_attn_fwd_rank(q, k, v, P, 0, out_fp32=True, out=parts,
                                                     lse=lp), max(3, reps // 4))
            emit(path, ms, acc.attention_flops(H, L, S, d), "TFLOP/s", "tensor",
                 form="per-step fp32 partials")
        elif path in ("factored_c4", "factored_c4_unfolded"):
            B, H, T, N, d, P = 1, 24, 48, 900, 128, 4
            # unfolded: the temporal ring as four 12-frame steps
            ra.ra_set_temporal_fold(path == "factored_c4")
            q, k, v = qkv(B, H, T * N, d)
            ws = torch.empty(ra.factored_attn_workspace(B, H, T, N, d), dtype=torch.uint8,
                             device="cuda")
            outs = (torch.empty_like(q), torch.empty((B, H, T * N), device="cuda"),
                    torch.empty_like(q), torch.empty((B, H, T * N), device="cuda"))
            ms = _time(lambda: ra.factored_attn(q, k, v, T, N, P, workspace=ws, outs=outs), reps)
            sp, tp = acc.factored_flops(B * H, T, N, d)
            ra.ra_set_temporal_fold(True)
            emit(path, ms, sp + tp, "TFLOP/s", "tensor", spatial_flops=sp, temporal_flops=tp)
        elif path.endswith("_c3") or path == "overlap_c3_stream":
            B, H, S, d, P = 1, 24, 14400, 128, 4
            q, k, v = qkv(B, H, S, d)
            fl = acc.attention_flops(B * H, S, S, d)
            if path in ("overlap_c3", "overlap_c3_stream"):
                ws = torch.empty(ra.ring_attn_fwd_overlap_workspace(B, H, S, d, P),
                                 dtype=torch.uint8, device="cuda")
                # overlap_c3: the exchange inside the step launches (no comm
                # stream); overlap_c3_stream: device copies on a comm stream
                comm = torch.cuda.Stream() if path == "overlap_c3_stream" else None
                ms = _time(lambda: ra.ring_attn_fwd_overlap(q, k, v, P, workspace=ws,
                                                            comm_stream=comm), reps)
                emit(path, ms, fl, "TFLOP/s", "tensor")
            elif path == "bwd_c3":
                o, lse = ra.ring_attn_fwd(q, k, v, P)
                g = _rand((B, H, S, d), gen)
                ws = torch.empty(ra.ring_attn_bwd_workspace(B, H, S), dtype=torch.uint8,
                                 device="cuda")
                grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
                ms = _time(lambda: ra.ring_attn_bwd(q, k, v, o, lse, g, P, workspace=ws,
                                                    grads=grads), reps)
                emit(path, ms, 2.5 * fl, "TFLOP/s", "tensor",
                     note="5 GEMMs per visible pair = 2.5x the forward")
            else:
                pr = [x.reshape(B, H, P, S // P, d).permute(2, 0, 1, 3, 4).contiguous()
                      for x in (q, k, v)]
                ws = torch.empty(max(ra.cp_variant_workspace(B, H, S, d, P),
                                     ra.ulysses_attn_workspace(B, H, S, d)),
                                 dtype=torch.uint8, device="cuda")
                fn = {"ulysses_c3": ra.ulysses_attn_fwd, "allgather_c3": ra.cp_allgather_attn_fwd,
                      "reducescatter_c3": ra.cp_reducescatter_attn_fwd}[path]
                ms = _time(lambda: fn(*pr, B, H, S, P, workspace=ws), reps)
                emit(path, ms, fl, "TFLOP/s", "tensor")
        else:
            raise SystemExit(f"unknown path {path}")
    if ra.ra_get_status() != 0:
        raise SystemExit("device watchdog fired")
    return out


ALL = ["shard", "transpose", "merge", "ring_c1", "ring_c2", "ring_c3", "rank_c5", "factored_c4",
       "factored_c4_unfolded", "overlap_c3", "overlap_c3_stream", "ulysses_c3", "allgather_c3",
       "reducescatter_c3", "bwd_c3"]


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--path", nargs="*", default=ALL)
    ap.add_argument("--reps", type=int, default=20)
    ap.add_argument("--graph", action="store_true",
                    help="also time the calls under CUDA-graph replay (graph_ms)")
    a = ap.parse_args()
    run(a.path, a.reps, a.graph)
