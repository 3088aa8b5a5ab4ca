"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds workload shapes, seeds and random-number draws only; it
contains none of the attention arithmetic.  Both sides import it; neither side
imports the other.

Workloads (tokens in global order, layout [B, H, S, d], d innermost):

  c1  non-causal ring,  B=1 H=2  S=1024   d=64  P=4 contiguous,          N(0,1),     seed 0
  c2  causal ring,      B=1 H=4  S=4096   d=64  P=2 zigzag (4 chunks),   N(0,1),     seed 1
  c3  video DiT,        B=1 H=24 S=14400  d=128 P=4 contiguous
      (16 frames x 900 tokens, 4 frames per chunk),                     N(0,1)*0.5, seed 2
  c4  factored video,   B=1 H=24 T=48 N=900 (S=43200) d=128, temporal ring
      P=4 chunks of 12 frames,                                          N(0,1),     seed 3
  c5  large video,      H=4 S=432000 (120 frames x 3600) d=128 P=8; one
      rank's 54,000 queries against all 8 KV blocks,                    N(0,1),     seed 4

The frame/token figures are the ones the "day 83" context-parallelism blog
works through ("What the numbers look like": 900 tokens per frame, 16 and 48
frames; 3,600 tokens x 120 frames = 432,000; CP=8 gives 54,000 per GPU).

Recipe: g = torch.Generator('cpu').manual_seed(seed); q, k, v drawn in that
order with torch.randn(shape, generator=g, dtype=float32); multiplied by the
workload's factor; rounded to bf16 (round-to-nearest-even, torch's cast).
Video token index = t * N + n (frame-major: whole frames are contiguous).
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    S: int            # global sequence length (all ranks)
    d: int
    P: int            # simulated ranks (ring size)
    causal: bool
    factor: float     # input scale
    seed: int
    T: int = 0        # frames (video workloads)
    N: int = 0        # tokens per frame (video workloads)
    q_rank: int = -1  # >= 0: only this rank's queries are generated (c5)

    @property
    def L(self) -> int:
        """Rows per rank chunk (S / P)."""
        return self.S // self.P

    @property
    def q_shape(self):
        rows = self.L if self.q_rank >= 0 else self.S
        return (self.B, self.H, rows, self.d)

    @property
    def kv_shape(self):
        return (self.B, self.H, self.S, self.d)


WORKLOADS = {
    "c1": Workload("c1", B=1, H=2, S=1024, d=64, P=4, causal=False, factor=1.0, seed=0),
    "c2": Workload("c2", B=1, H=4, S=4096, d=64, P=2, causal=True, factor=1.0, seed=1),
    "c3": Workload("c3", B=1, H=24, S=14400, d=128, P=4, causal=False, factor=0.5, seed=2,
                   T=16, N=900),
    "c4": Workload("c4", B=1, H=24, S=43200, d=128, P=4, causal=False, factor=1.0, seed=3,
                   T=48, N=900),
    "c5": Workload("c5", B=1, H=4, S=432000, d=128, P=8, causal=False, factor=1.0, seed=4,
                   T=120, N=3600, q_rank=0),
}


def _draw(shape, g, factor):
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    if factor != 1.0:
        x.mul_(factor)
    return x.to(torch.bfloat16)


def make_qkv(w: Workload | str):
    """Return (q, k, v) as contiguous bf16 CPU tensors in global token order."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    g = torch.Generator("cpu").manual_seed(w.seed)
    q = _draw(w.q_shape, g, w.factor)
    k = _draw(w.kv_shape, g, w.factor)
    v = _draw(w.kv_shape, g, w.factor)
    return q, k, v


def make_custom(shape_q, shape_kv, seed, factor=1.0):
    """Seeded bf16 (q, k, v) for ad-hoc test shapes, same recipe as the workloads."""
    g = torch.Generator("cpu").manual_seed(seed)
    q = _draw(tuple(shape_q), g, factor)
    k = _draw(tuple(shape_kv), g, factor)
    v = _draw(tuple(shape_kv), g, factor)
    return q, k, v


def make_partials(n, rows, d, seed, empty_rows=0, empty_parts=0, o_scale=0.25):
    """Seeded fp32 partial outputs and log-sum-exps for merge tests.

    Returns o [n, rows, d] fp32 and lse [n, rows] fp32.  The first `empty_rows`
    rows have every partial empty (lse = -inf, o = 0); in the next rows, the
    first `empty_parts` partials are empty.  Everything else is N(0, o_scale^2)
    for o (a normalised attention output is a convex combination of value rows,
    so its entries are small) and N(0, 2^2) for lse.
    """
    g = torch.Generator("cpu").manual_seed(seed)
    o = torch.randn((n, rows, d), generator=g, dtype=torch.float32) * o_scale
    lse = torch.randn((n, rows), generator=g, dtype=torch.float32) * 2.0
    if empty_rows:
        o[:, :empty_rows] = 0.0
        lse[:, :empty_rows] = float("-inf")
    if empty_parts:
        lo, hi = empty_rows, min(rows, empty_rows + max(1, rows // 4))
        o[:empty_parts, lo:hi] = 0.0
        lse[:empty_parts, lo:hi] = float("-inf")
    return o.contiguous(), lse.contiguous()


def sample_rows(w: Workload | str, per_head: int, index: int | None = None):
    """Query rows (per head, global order) for sampled parity on large workloads.

    The first and last row of every rank chunk, then seeded-uniform rows
    (seed 1000 + workload index) until `per_head` distinct rows are chosen.
    For workloads that generate one rank's queries only, rows are local to it.
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    if index is None:
        index = int(w.name[1:]) if w.name[1:].isdigit() else 0
    n_rows = w.q_shape[2]
    chunks = 1 if w.q_rank >= 0 else w.P
    L = n_rows // chunks
    fixed = []
    for r in range(chunks):
        fixed += [r * L, r * L + L - 1]
    rng = np.random.default_rng(1000 + index)
    chosen = list(dict.fromkeys(fixed))
    while len(chosen) < per_head:
        c = int(rng.integers(0, n_rows))
        if c not in chosen:
            chosen.append(c)
    return np.array(sorted(chosen[:per_head]), dtype=np.int64)


def tile_rows(n_heads: int, n_rows: int, chunk: int, tile: int = 128, salt: int = 0):
    """Flat row indices (head * n_rows + row) with one row in every `tile`-row
    query tile of every `chunk`-row chunk of every head.

    Tile t of chunk c in head h contributes row c*chunk + t*tile + lane, with
    lane = (37*t + 53*h + 11*c + salt) mod (rows of that tile), so that over
    the tiles every lane position of a full tile is met, and a short last tile
    contributes a different one of its rows per chunk and head.
    """
    out = []
    n_chunks = n_rows // chunk
    n_t = (chunk + tile - 1) // tile
    for h in range(n_heads):
        for c in range(n_chunks):
            t = np.arange(n_t, dtype=np.int64)
            rows_in_tile = np.minimum(tile, chunk - t * tile)
            lane = (37 * t + 53 * h + 11 * c + salt) % rows_in_tile
            r = t * tile + lane
            out.append(h * n_rows + c * chunk + r)
    return np.unique(np.concatenate(out)) if out else np.empty(0, dtype=np.int64)
