"""Pure-Python brute-force attention for tiny shapes: TEST INFRASTRUCTURE ONLY.

An independent restatement of the full-attention definition (ultralytics
glossary "Context Parallelism", "How Context Parallelism Works": the ring
result equals full-sequence attention), written without the max shift that
the C oracle uses, so a mistake in either one shows up as a mismatch:

    w_ij = exp((q_i . k_j) / sqrt(d))     for j in K(i)
    LSE_i = log(sum_j w_ij)
    O_i   = sum_j w_ij v_j / sum_j w_ij

K(i) is every key, or {j <= i} when causal.  Inputs must be small enough that
exp() does not overflow (|score| well below 700).
"""
from __future__ import annotations

import math


def attention(q, k, v, causal=False):
    """q, k, v: nested lists [S][d] of floats (one head).  Returns (O, LSE)."""
    S, d = len(q), len(q[0])
    Sk = len(k)
    inv = 1.0 / math.sqrt(d)
    O, LSE = [], []
    for i in range(S):
        keys = range(min(i + 1, Sk)) if causal else range(Sk)
        w = []
        for j in keys:
            w.append(math.exp(sum(q[i][c] * k[j][c] for c in range(d)) * inv))
        z = sum(w)
        O.append([sum(w[t] * v[j][c] for t, j in enumerate(keys)) / z for c in range(d)])
        LSE.append(math.log(z))
    return O, LSE
