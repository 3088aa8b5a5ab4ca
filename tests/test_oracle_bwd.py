"""Pins for the oracle's attention gradients (fp64)."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import brute


def _loss(q, k, v, w, causal):
    """sum_i O_i . w_i with the pure-Python brute force (one head)."""
    O, _ = brute.attention(q, k, v, causal)
    return sum(O[i][c] * w[i][c] for i in range(len(O)) for c in range(len(O[0])))


@pytest.mark.parametrize("causal", [False, True])
def test_finite_differences_against_brute_force(causal):
    S, d = 5, 4
    q, k, v = synth.make_custom((1, 1, S, d), (1, 1, S, d), seed=900 + causal)
    w, _, _ = synth.make_custom((1, 1, S, d), (1, 1, 1, 1), seed=901)
    dq, dk, dv = oracle.attention_bwd(q, k, v, w, causal=causal)
    Q, K, V, W = (x[0, 0].double().tolist() for x in (q, k, v, w))
    h = 1e-6
    for name, X, G in (("q", Q, dq), ("k", K, dk), ("v", V, dv)):
        for i in range(S):
            for c in range(d):
                plus = [row[:] for row in X]
                minus = [row[:] for row in X]
                plus[i][c] += h
                minus[i][c] -= h
                args_p = {"q": Q, "k": K, "v": V}
                args_m = dict(args_p)
                args_p[name], args_m[name] = plus, minus
                num = (_loss(args_p["q"], args_p["k"], args_p["v"], W, causal)
                       - _loss(args_m["q"], args_m["k"], args_m["v"], W, causal)) / (2 * h)
                assert abs(num - G[0, 0, i, c]) <= 1e-7, (name, i, c, num, G[0, 0, i, c])


@pytest.mark.parametrize("causal", [False, True])
def test_against_torch_float64_autograd(causal):
    S, d = 192, 32
    q, k, v = synth.make_custom((1, 2, S, d), (1, 2, S, d), seed=902)
    w, _, _ = synth.make_custom((1, 2, S, d), (1, 1, 1, 1), seed=903)
    dq, dk, dv = oracle.attention_bwd(q, k, v, w, causal=causal)
    Q, K, V = (x.double().requires_grad_() for x in (q, k, v))
    s = Q @ K.transpose(-1, -2) / math.sqrt(d)
    if causal:
        s = s.masked_fill(torch.triu(torch.ones(S, S, dtype=torch.bool), 1), float("-inf"))
    O = torch.softmax(s, -1) @ V
    O.backward(w.double())
    for ours, ref in ((dq, Q.grad), (dk, K.grad), (dv, V.grad)):
        assert np.max(np.abs(ours - ref.numpy())) <= 1e-11


def test_key_gradients_sum_to_zero_and_value_shift_invariance():
    S, d = 40, 8
    q, k, v = synth.make_custom((1, 2, S, d), (1, 2, S, d), seed=904)
    w, _, _ = synth.make_custom((1, 2, S, d), (1, 1, 1, 1), seed=905)
    # values on a 1/8 grid, so that v + 1/2 is exact in bf16
    v = (torch.round(v.float() * 8) / 8).to(torch.bfloat16)
    for causal in (False, True):
        dq, dk, dv = oracle.attention_bwd(q, k, v, w, causal=causal)
        # sum_j dS_ij = 0 for every query, so the key gradients sum to zero
        assert np.max(np.abs(dk.sum(axis=2))) <= 1e-12
        # adding a constant row c to every value shifts O by c and leaves dQ, dK
        v2 = (v.float() + torch.tensor([0.5] * d)).to(torch.bfloat16)
        dq2, dk2, dv2 = oracle.attention_bwd(q, k, v2, w, causal=causal)
        assert np.max(np.abs(dq2 - dq)) <= 1e-12 and np.max(np.abs(dk2 - dk)) <= 1e-12
        assert np.max(np.abs(dv2 - dv)) <= 1e-12


def test_zero_upstream_gradient_gives_zero():
    q, k, v = synth.make_custom((1, 1, 16, 8), (1, 1, 16, 8), seed=906)
    z = torch.zeros((1, 1, 16, 8), dtype=torch.bfloat16)
    for g in oracle.attention_bwd(q, k, v, z, causal=True):
        assert np.all(g == 0.0)
