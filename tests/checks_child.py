"""Child process of tests/test_gpu_checks.py: runs small cases of every entry
point on the library named by RINGATTN_LIB (the RA_CHECKS build), checks each
against the fp64 oracle and requires the device status word to stay 0 (no
bounds check failed, no wait expired).  Prints "ok" on success."""
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402
import ring_attention_attn_gb300 as ra  # noqa: E402


def _close(o, l, ro, rl):
    o = o.double().cpu().numpy().reshape(ro.shape)
    l = l.double().cpu().numpy().reshape(rl.shape)
    fin = np.isfinite(rl)
    assert np.array_equal(fin, np.isfinite(l))
    assert np.max(np.abs(o - ro)) <= 1e-2, np.max(np.abs(o - ro))
    assert np.max(np.abs(l[fin] - rl[fin])) <= 1e-3


def _status(what):
    s = ra.ra_get_status()
    assert s == 0, f"{what}: device status {s}"


def main():
    assert ra.ra_checks_enabled(), "RINGATTN_LIB does not name the RA_CHECKS build"
    # the reporting path itself
    ra.ra_checks_selftest()
    assert ra.ra_get_status() == -7
    assert ra.ra_get_status() == 0
    # ring forward, c1 (contiguous) and c2 (causal zigzag), through the shard kernel
    for name in ("c1", "c2"):
        w = synth.WORKLOADS[name]
        q, k, v = synth.make_qkv(w)
        layout = 1 if w.causal else 0
        qs, ks, vs = (ra.ra_cp_shard(x.cuda(), w.P, layout) for x in (q, k, v))
        o, l = ra.ring_attn_fwd(qs, ks, vs, w.P, causal=w.causal)
        o = ra.ra_cp_shard(o, w.P, layout, inverse=True)
        _, g2s = oracle.shard_index(w.S, w.P, layout)
        l = l.cpu()[:, :, torch.from_numpy(g2s)]
        _status(name)
        ro, rl = oracle.attention(q, k, v, causal=w.causal)
        _close(o, l, ro, rl)
    # stacked last rows, per-step partials + merge, overlap, CP forms
    B, H, S, d, P = 1, 4, 1088, 128, 4  # Ulysses needs H % P == 0
    q, k, v = synth.make_custom((B, H, S, d), (B, H, S, d), seed=5)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    ro, rl = oracle.attention(q, k, v)
    o, l = ra.ring_attn_fwd(qd, kd, vd, P)
    _status("stacked")
    _close(o, l, ro, rl)
    L = S // P
    parts, lp = ra.ring_attn_fwd_rank(qd[:, :, :L].contiguous(), kd, vd, P, 0, out_fp32=True)
    mo, ml = ra.lse_merge(parts, lp)
    _status("partials + merge")
    _close(mo, ml, ro[:, :, :L], rl[:, :, :L])
    o, l = ra.ring_attn_fwd_overlap(qd, kd, vd, P, comm_stream=torch.cuda.Stream())
    _status("overlap")
    _close(o, l, ro, rl)
    per_rank = [x.reshape(B, H, P, L, d).permute(2, 0, 1, 3, 4).contiguous() for x in (qd, kd, vd)]
    for fn in (ra.ulysses_attn_fwd, ra.cp_allgather_attn_fwd, ra.cp_reducescatter_attn_fwd):
        o, l = fn(*per_rank, B, H, S, P)
        _status(fn.__name__)
        _close(o.permute(1, 2, 0, 3, 4).reshape(B, H, S, d),
               l.permute(1, 2, 0, 3).reshape(B, H, S), ro, rl)
    # factored: packed temporal (in place) and chunks over 128 frames (transposes)
    for (T, N, dd, PP) in ((24, 30, 128, 4), (260, 3, 64, 2)):
        q, k, v = synth.make_custom((1, 2, T * N, dd), (1, 2, T * N, dd), seed=T)
        outs = ra.factored_attn(q.cuda(), k.cuda(), v.cuda(), T, N, PP)
        _status(f"factored T={T}")
        for which, (o, l) in (("spatial", outs[:2]), ("temporal", outs[2:])):
            _close(o, l, *oracle.factored(q, k, v, T, N, which))
    # backward, non-causal with stacked rows and causal
    for causal, S2 in ((False, 1088), (True, 1024)):
        q, k, v = synth.make_custom((1, 2, S2, 128), (1, 2, S2, 128), seed=S2)
        g = synth.make_custom((1, 2, S2, 128), (1, 1, 1, 1), seed=S2 + 1)[0]
        lay = 1 if causal else 0
        qs, ks, vs, gs = (ra.ra_cp_shard(x.cuda(), 4, lay) for x in (q, k, v, g))
        o, l = ra.ring_attn_fwd(qs, ks, vs, 4, causal=causal)
        dq, dk, dv = ra.ring_attn_bwd(qs, ks, vs, o, l, gs, 4, causal=causal)
        _status(f"backward causal={causal}")
        want = oracle.attention_bwd(q, k, v, g, causal=causal)
        for got, ref in zip((dq, dk, dv), want):
            got = ra.ra_cp_shard(got, 4, lay, inverse=True).double().cpu().numpy()
            assert np.max(np.abs(got - ref)) <= 1e-2 * np.max(np.abs(ref)) + 1e-3
    print("ok")


if __name__ == "__main__":
    main()
