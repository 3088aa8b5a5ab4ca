"""Seeded random shapes through the ring and factored entry points against the
oracle: ragged chunk lengths, odd head counts, both head sizes, causal and
not, P from 1 to 8, frame counts around the 16/32/128-row packing limits and
the folding of short rank chunks."""
import numpy as np
import pytest
import torch

import oracle
import synth
import ring_attention_attn_gb300 as ra

pytestmark = pytest.mark.gpu

O_TOL = 1e-2
LSE_TOL = 1e-3
# bf16 keeps 8 significant bits: rounding the output O to bf16 alone moves it
# by up to half a unit in the last place, 2^-9 |O|.  On the five workloads
# |O| stays small and the plain 1e-2 bound holds; a row that sees one to a
# few keys (4-token sequences, 1-frame chunks) has |O| up to ~4, where that
# rounding reaches 1e-2 by itself.  These random shapes therefore allow one
# bf16 unit of |O| on top of the bound.
O_REL = 2.0 ** -8


def _cmp(o_gpu, l_gpu, o_ref, l_ref):
    o = o_gpu.double().cpu().numpy().reshape(o_ref.shape)
    l = l_gpu.double().cpu().numpy().reshape(l_ref.shape)
    fin = np.isfinite(l_ref)
    assert np.array_equal(fin, np.isfinite(l))
    excess = np.abs(o - o_ref) - (O_TOL + O_REL * np.abs(o_ref))
    assert np.max(excess) <= 0, f"max|dO| = {np.max(np.abs(o - o_ref)):.3e}"
    if fin.any():
        assert np.max(np.abs(l[fin] - l_ref[fin])) <= LSE_TOL


def _ring_cases():
    rng = np.random.default_rng(20261202)
    cases = []
    while len(cases) < 24:
        P = int(rng.integers(1, 9))
        causal = bool(rng.integers(0, 2))
        unit = 2 * P if causal else P
        S = unit * int(rng.integers(1, max(2, 2400 // unit)))
        cases.append((1, int(rng.integers(1, 4)), S, int(rng.choice([64, 128])), P, causal,
                      int(rng.integers(0, 1 << 30))))
    return cases


@pytest.mark.parametrize("B,H,S,d,P,causal,seed", _ring_cases())
def test_ring_random_shapes(B, H, S, d, P, causal, seed):
    layout = 1 if causal else 0
    q, k, v = synth.make_custom((B, H, S, d), (B, H, S, d), seed=seed)
    s2g, g2s = oracle.shard_index(S, P, layout)
    idx, inv = torch.from_numpy(s2g), torch.from_numpy(g2s)
    qs, ks, vs = (x[:, :, idx].contiguous().cuda() for x in (q, k, v))
    out, lse = ra.ring_attn_fwd(qs, ks, vs, P, causal=causal)
    torch.cuda.synchronize()
    assert ra.ra_get_status() == 0
    o = out.cpu()[:, :, inv]
    l = lse.cpu()[:, :, inv]
    ro, rl = oracle.attention(q, k, v, causal=causal)
    _cmp(o, l, ro, rl)


def _factored_cases():
    rng = np.random.default_rng(4242)
    cases = []
    # (8, 8), (36, 6), (48, 8), (60, 4): short chunks that fold by 4, 3, 4, 2.
    for T, P in [(4, 4), (15, 5), (16, 1), (17, 1), (32, 2), (33, 3), (64, 2), (96, 3), (128, 1),
                 (130, 2), (8, 8), (36, 6), (48, 8), (60, 4)]:
        N = int(rng.integers(3, 60))
        cases.append((1, int(rng.integers(1, 3)), T, N, int(rng.choice([64, 128])), P,
                      int(rng.integers(0, 1 << 30))))
    return cases


@pytest.mark.parametrize("B,H,T,N,d,P,seed", _factored_cases())
def test_factored_random_shapes(B, H, T, N, d, P, seed):
    q, k, v = synth.make_custom((B, H, T * N, d), (B, H, T * N, d), seed=seed)
    os_, ls, ot, lt = ra.factored_attn(q.cuda(), k.cuda(), v.cuda(), T, N, P)
    torch.cuda.synchronize()
    assert ra.ra_get_status() == 0
    ro, rl = oracle.factored(q, k, v, T, N, "spatial")
    _cmp(os_, ls, ro, rl)
    ro, rl = oracle.factored(q, k, v, T, N, "temporal")
    _cmp(ot, lt, ro, rl)
