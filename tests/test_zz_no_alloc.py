"""factored_attn_static: the entry point for callers that may not allocate
device memory (e.g. their device memory is all owned by a pool set up at
start-up, or an allocation is not allowed where they call the library).

It runs the same kernels on the same scratch layout as factored_attn with a
caller workspace, so its outputs must be bit-identical to factored_attn's, on
two calls in a row (the second call reuses the fixed scratch the first one
left behind); one case is also checked against the fp64 oracle.  It must
refuse sizes its fixed scratch cannot hold, and accept any size whose rank
chunks run in place.  This file is collected last so that a run stopping at
the first failure has run every other test first; it also passes alone in a
fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
import ring_attention_attn_gb300 as ra
from ring_attention_attn_gb300 import _abi

pytestmark = pytest.mark.gpu

O_TOL = 1e-2
LSE_TOL = 1e-3
STATIC_SCRATCH_BYTES = 64 << 20  # RA_STATIC_SCRATCH_BYTES in include/ringattn.h


def _outs(B, H, S, d):
    return (torch.empty((B, H, S, d), dtype=torch.bfloat16, device="cuda"),
            torch.empty((B, H, S), dtype=torch.float32, device="cuda"),
            torch.empty((B, H, S, d), dtype=torch.bfloat16, device="cuda"),
            torch.empty((B, H, S), dtype=torch.float32, device="cuda"))


def _call_static(q, k, v, T, N, P, outs):
    """Calls the C entry point directly through ctypes."""
    B, H, S, d = q.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return _abi.lib().factored_attn_static(p(q), p(k), p(v), p(outs[0]), p(outs[1]), p(outs[2]),
                                           p(outs[3]), B, H, T, N, d, P, stream)


def _same_bits(a, b):
    return torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                       b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))


def _cmp_oracle(got, want_o, want_l, rows, d):
    o = got[0].reshape(-1, d)[rows].double().cpu().numpy()
    l = got[1].reshape(-1)[rows].double().cpu().numpy()
    assert np.max(np.abs(o - want_o)) <= O_TOL
    assert np.max(np.abs(l - want_l)) <= LSE_TOL


@pytest.mark.parametrize("B,H,T,N,d,P,seeds", [(1, 2, 8, 50, 64, 4, (11, 12)),
                                               (1, 3, 12, 130, 128, 4, (21, 22)),
                                               # chunks over 128 frames: the scratch is used
                                               (1, 1, 260, 3, 64, 2, (31, 32)),
                                               (1, 2, 136, 5, 128, 1, (41, 42)),
                                               # T > 128 but 128-frame chunks: run in place,
                                               # although factored_attn_workspace (any P)
                                               # would exceed the fixed scratch
                                               (1, 2, 256, 900, 128, 2, (51, 52))])
def test_static_scratch_matches_workspace_version_twice(B, H, T, N, d, P, seeds):
    S = T * N
    big = ra.factored_attn_workspace(B, H, T, N, d) > STATIC_SCRATCH_BYTES
    assert big == (T == 256)
    for seed in seeds:  # two calls in a row, different inputs
        q, k, v = (x.cuda() for x in synth.make_custom((B, H, S, d), (B, H, S, d), seed=seed))
        got = _outs(B, H, S, d)
        assert _call_static(q, k, v, T, N, P, got) == 0
        want = ra.factored_attn(q, k, v, T, N, P)
        torch.cuda.synchronize()
        assert ra.ra_get_status() == 0
        for g, w in zip(got, want):
            assert _same_bits(g, w)
        if seed == seeds[1] and T == 260:
            # the second call, on the scratch the first one left, against the oracle
            qc, kc, vc = (x.cpu() for x in (q, k, v))
            rows = np.arange(B * H * S)
            ro, rl = oracle.factored(qc, kc, vc, T, N, "spatial")
            _cmp_oracle(got[0:2], ro.reshape(-1, d), rl.reshape(-1), rows, d)
            ro, rl = oracle.factored(qc, kc, vc, T, N, "temporal")
            _cmp_oracle(got[2:4], ro.reshape(-1, d), rl.reshape(-1), rows, d)


def test_static_scratch_refuses_sizes_beyond_its_limit():
    B, H, T, N, d, P = 1, 24, 256, 900, 128, 1  # 256-frame chunks: ~5.7 GB of scratch
    assert ra.factored_attn_workspace(B, H, T, N, d) > STATIC_SCRATCH_BYTES
    x = torch.empty((1, 1, 1, d), dtype=torch.bfloat16, device="cuda")  # never touched
    lse = torch.empty((1,), dtype=torch.float32, device="cuda")
    p = ctypes.c_void_p
    rc = _abi.lib().factored_attn_static(p(x.data_ptr()), p(x.data_ptr()), p(x.data_ptr()),
                                         p(x.data_ptr()), p(lse.data_ptr()), p(x.data_ptr()),
                                         p(lse.data_ptr()), B, H, T, N, d, P,
                                         p(torch.cuda.current_stream().cuda_stream))
    assert rc == -6  # RA_ERR_WORKSPACE


CHILD = r"""
import sys
sys.path.insert(0, {root!r})
import torch
import ring_attention_attn_gb300 as ra

def free():
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]

def args(T, N, d=64):
    S = T * N
    q, k, v = (torch.randn(1, 2, S, d, device="cuda").bfloat16() for _ in range(3))
    outs = (torch.empty_like(q), torch.empty(1, 2, S, device="cuda"),
            torch.empty_like(q), torch.empty(1, 2, S, device="cuda"))
    return q, k, v, outs

small = args(8, 50)    # T / P = 2 frames per chunk: no scratch
big = args(260, 3)     # T / P = 130: the scratch is used
# the attention kernels (and the workspace version's buffers) first
ra.factored_attn(*small[:3], 8, 50, 4, outs=small[3])
ra.factored_attn(*big[:3], 260, 3, 2, outs=big[3])
f0 = free()
ra.factored_attn_static(*small[:3], 8, 50, 4, small[3])
f1 = free()
ra.factored_attn_static(*big[:3], 260, 3, 2, big[3])
f2 = free()
assert ra.ra_get_status() == 0
print(f0 - f1, f1 - f2)
"""


def test_scratch_is_placed_only_by_calls_that_need_it():
    """Under the runtime's default lazy loading, a call whose rank chunks fit
    one tile does not make the 64 MiB array resident; the first call that
    needs scratch does.  Run in a fresh process, so that no earlier call in
    this session has placed the array already."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, CUDA_MODULE_LOADING="LAZY")
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=root)], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    no_scratch, with_scratch = (int(x) for x in r.stdout.split()[-2:])
    mib = 1 << 20
    assert no_scratch < 16 * mib, no_scratch
    assert with_scratch >= 60 * mib, with_scratch
