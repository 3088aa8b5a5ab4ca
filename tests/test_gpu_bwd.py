"""GPU parity of the backward pass against the fp64 oracle gradients.

Tolerance: bf16 inputs, P and dS rounded to bf16 before their MMAs, fp32
accumulation, bf16 gradients; each gradient must satisfy
max|g_gpu - g_ref| <= 1e-2 * max|g_ref| + 1e-3 (measured: about 4e-3 * max).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import ring_attention_attn_gb300 as ra

pytestmark = pytest.mark.gpu


def _shard(x, P, layout):
    s2g, _ = oracle.shard_index(x.shape[2], P, layout)
    return x[:, :, torch.from_numpy(s2g)].contiguous()


def _unshard(y, P, layout):
    _, g2s = oracle.shard_index(y.shape[2], P, layout)
    return y[:, :, torch.from_numpy(g2s)].contiguous()


CASES = [
    (1, 2, 512, 64, 2, False),
    (1, 2, 1024, 128, 4, False),
    (1, 2, 1024, 64, 2, True),
    (2, 1, 600, 128, 3, True),
    (1, 1, 256, 128, 1, True),
    (1, 3, 1000, 128, 4, False),
    (1, 1, 16, 64, 8, True),
    (1, 2, 1088, 128, 4, False),  # 272-row chunks: the ranks' last 16 rows stacked
    (1, 1, 504, 64, 3, False),    # 168-row chunks: 3 x 40 rows stacked
    # a longer ring: 1,040-row chunks (9 tiles each, the last 16 rows of every
    # chunk stacked), 16 heads so the oracle (parallel over heads) uses 16 cores
    (1, 16, 4160, 128, 4, False),
]


@pytest.mark.parametrize("B,H,S,d,P,causal", CASES)
def test_ring_backward_matches_oracle(B, H, S, d, P, causal):
    layout = 1 if causal else 0
    q, k, v = synth.make_custom((B, H, S, d), (B, H, S, d), seed=S + d + P + 7 * causal)
    g, _, _ = synth.make_custom((B, H, S, d), (1, 1, 1, 1), seed=S + 3)
    qs, ks, vs, gs = (_shard(x, P, layout).cuda() for x in (q, k, v, g))
    out, lse = ra.ring_attn_fwd(qs, ks, vs, P, causal=causal)
    dq, dk, dv = ra.ring_attn_bwd(qs, ks, vs, out, lse, gs, P, causal=causal)
    torch.cuda.synchronize()
    assert ra.ra_get_status() == 0
    ref = oracle.attention_bwd(q, k, v, g, causal=causal)
    for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        got = _unshard(got.cpu(), P, layout).double().numpy()
        err = np.max(np.abs(got - want))
        scale = np.max(np.abs(want))
        assert err <= 1e-2 * scale + 1e-3, f"{name}: max|d| = {err:.3e}, max|ref| = {scale:.3e}"


def _random_cases():
    """Seeded random ring shapes for the backward: P from 1 to 8, causal or
    not, both head sizes, ragged chunks.  RA_FUZZ_SCALE / RA_FUZZ_SEED /
    RA_FUZZ_SMAX widen them as in tests/test_gpu_fuzz.py."""
    import os
    scale = int(os.environ.get("RA_FUZZ_SCALE", "1"))
    smax = int(os.environ.get("RA_FUZZ_SMAX", "2400"))
    rng = np.random.default_rng(5150 + int(os.environ.get("RA_FUZZ_SEED", "0")))
    cases = []
    while len(cases) < 8 * scale:
        P = int(rng.integers(1, 9))
        causal = bool(rng.integers(0, 2))
        unit = 2 * P if causal else P
        S = unit * int(rng.integers(1, max(2, min(smax, 1600) // unit)))
        cases.append((1, int(rng.integers(1, 3)), S, int(rng.choice([64, 128])), P, causal))
    return cases


@pytest.mark.parametrize("B,H,S,d,P,causal", _random_cases())
def test_ring_backward_random_shapes(B, H, S, d, P, causal):
    test_ring_backward_matches_oracle(B, H, S, d, P, causal)
